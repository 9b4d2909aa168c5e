"""GPU parity of NVFP4 expert bundles (E2M1 codes, E4M3 block scales of 16 k, fp32 matrix
scales) against the fp64 oracle, through the C ABI: the grouped SwiGLU on its own, whole
layers with a shared expert (routed and shared groups in one tcgen05 launch, each with its own
bundle layout), the full Qwen1.5-MoE shape, every E4M3 scale byte, and the negative test of
bundle atomicity (foreign matrix scales).
Tolerance as for the other formats: max |err| <= 2e-2 max |ref|, sum |err| / sum |ref| <= 5e-3.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import bf16, moe_ref

from gpu_util import assert_close, check_ids, spread_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import expert_dispatch_streaming_gb300 as m
    return m


@pytest.fixture(scope="module")
def syn(moe):
    from expert_dispatch_streaming_gb300 import synthetic
    return synthetic


SMALL = [
    wl.custom("fp4small", cfg_id=160, H=256, E=16, k=4, I=384, gating="softmax_renorm",
              wdtype="nvfp4"),
    wl.custom("fp4qwenlike", cfg_id=161, H=512, E=60, k=4, I=256, gating="softmax", Is=384,
              shared_gate="sigmoid", zipf_s=1.0, bias_kind="logit", wdtype="nvfp4"),
    wl.custom("fp4dslike", cfg_id=162, H=512, E=64, k=8, I=256, gating="sigmoid_bias_renorm",
              scale=2.5, Is=256, shared_gate="one", zipf_s=1.1, bias_kind="select",
              wdtype="nvfp4"),
]


def _grouped(moe, syn, cfg, xb, offsets, src_rows, bundles):
    rows = int(offsets[-1])
    x_perm = torch.from_numpy(np.ascontiguousarray(xb.view(np.int16)[src_rows])).cuda()
    off = torch.from_numpy(np.asarray(offsets, np.int32)).cuda()
    y = torch.zeros((rows, cfg.H), dtype=torch.int16, device="cuda")
    nws = moe.moe_grouped_swiglu_workspace_size(rows, len(bundles), cfg.H, cfg.I, "nvfp4")
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    moe.moe_grouped_swiglu(x_perm, off, bundles, len(bundles), cfg.H, cfg.I, "nvfp4", rows, y,
                           ws, nws)
    torch.cuda.synchronize()
    return y.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
@pytest.mark.parametrize("T", [1, 57, 300])
def test_grouped_swiglu_nvfp4(moe, syn, cfg, T):
    rng = np.random.default_rng(T + cfg.cfg_id)
    xb = wl.tokens(cfg, T)
    ids = np.stack([rng.choice(cfg.E, cfg.k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, pos, src = moe_ref.dispatch(ids, cfg.E)
    dl = syn.DeviceLayer(cfg)
    y = _grouped(moe, syn, cfg, xb, offsets, src // cfg.k, [dl.routed[e] for e in range(cfg.E)])
    x = bf16.decode(xb)
    ref = np.zeros((T * cfg.k, cfg.H))
    for e in range(cfg.E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            wg, wu, wd = moe_ref.expert_matrices(wl.expert(cfg, 0, e))
            ref[lo:hi], _ = moe_ref.swiglu_ffn(x[src[lo:hi] // cfg.k], wg, wu, wd)
    assert_close(y, ref, f"{cfg.name} T={T} y_perm")


def _layer_case(syn, cfg, T, rows=None):
    dl = syn.DeviceLayer(cfg)
    xb = wl.tokens(cfg, T)
    x = syn.to_device_bits(xb)
    ws = dl.workspace(T)
    ids = torch.empty((T, cfg.k), dtype=torch.int32, device="cuda")
    out, _ = dl.forward(x, ws, ids_out=ids)
    out2, _ = dl.forward(x, ws)
    torch.cuda.synchronize()
    got = syn.bits_of(out)
    assert np.array_equal(got, syn.bits_of(out2)), "second run differs (nondeterminism)"
    ids = ids.cpu().numpy()
    check_ids(cfg, ids, None, xb)
    if isinstance(rows, str) and rows == "spread":
        rows = spread_rows(ids, cfg.E)
    ref = moe_ref.layer_forward(cfg, 0, xb, forced_ids=ids, rows=rows)
    return assert_close(got[ref["rows"]], ref["out"], f"{cfg.name} T={T}")


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
@pytest.mark.parametrize("T", [1, 16, 133])
def test_layer_forward_nvfp4_small(syn, cfg, T):
    _layer_case(syn, cfg, T)


@pytest.mark.parametrize("T", [1, 16, 256, 2048, 8192])
def test_layer_forward_qwen_nvfp4(syn, T):
    """The full Qwen1.5-MoE shape with NVFP4 experts (routed and shared); sampled rows."""
    _layer_case(syn, wl.QWEN_NVFP4, T, rows="spread")


def test_every_e4m3_scale_byte(moe, syn):
    """Down-projection column n of a single expert uses block scale byte n (0x00 .. 0x7E, all
    127 valid E4M3 values incl. the subnormals, plus 0x38 for the last column) in every block,
    so each output column is checked against the oracle relative to its own magnitude."""
    H, I = 128, 256
    cfg = wl.custom("fp4bytes", cfg_id=163, H=H, E=1, k=1, I=I, wdtype="nvfp4")
    w = wl.expert(cfg, 0, 0)
    sd = np.tile(np.minimum(np.arange(H), 0x7E).astype(np.uint8), (I // 16, 1))
    sd[:, H - 1] = 0x38
    gs = np.array([w.gs[0], w.gs[1], 1.0], np.float32)
    nb = moe.moe_bundle_bytes(H, I, "nvfp4")
    host = np.zeros(nb, np.uint8)
    moe.moe_pack_bundle_nvfp4(H, I, w.wg, w.wu, w.wd, w.sg, w.su, sd, gs, host)
    dev = torch.from_numpy(host).cuda()
    T = 40
    xb = wl.tokens(cfg, T)
    y = _grouped(moe, syn, cfg, xb, [0, T], np.arange(T), [dev])
    ew = wl.ExpertWeights("nvfp4", w.wg, w.wu, w.wd, w.sg, w.su, sd, gs)
    wg, wu, wd = moe_ref.expert_matrices(ew)
    ref, _ = moe_ref.swiglu_ffn(bf16.decode(xb), wg, wu, wd)
    got = bf16.decode(y)
    assert np.all(got[:, 0] == 0) and np.all(ref[:, 0] == 0)            # scale 0: zero column
    for n in range(1, H):
        col = np.abs(ref[:, n]).max()
        err = np.abs(got[:, n] - ref[:, n]).max()
        assert err <= 2e-2 * col, f"column {n} (scale byte {sd[0, n]:#x}): {err} vs {col}"


def test_nvfp4_bundle_with_foreign_matrix_scales_fails_parity(moe, syn):
    """The matrix scales travel inside the bundle: bundles whose 12-byte matrix-scale block
    comes from another expert give a wrong layer."""
    cfg = SMALL[0]
    hb = syn.host_bundles(cfg, 0, list(range(cfg.E)), pinned=False)
    lay = moe.bundle_layout(cfg.H, cfg.I, cfg.wdtype)
    g0 = lay.global_scale_offset
    bad = hb.clone()
    for e in range(cfg.E):
        bad[e, g0:g0 + 12] = hb[(e + 5) % cfg.E, g0:g0 + 12]
    T = 33
    xb = wl.tokens(cfg, T)
    x = syn.to_device_bits(xb)
    good_l = syn.DeviceLayer(cfg, bundles_override=hb)
    bad_l = syn.DeviceLayer(cfg, bundles_override=bad)
    ws = good_l.workspace(T)
    ids = torch.empty((T, cfg.k), dtype=torch.int32, device="cuda")
    o1, _ = good_l.forward(x, ws, ids_out=ids)
    o2, _ = bad_l.forward(x, ws)
    torch.cuda.synchronize()
    ref = moe_ref.layer_forward(cfg, 0, xb, forced_ids=ids.cpu().numpy())
    assert_close(syn.bits_of(o1), ref["out"], "good bundles")
    with pytest.raises(AssertionError):
        assert_close(syn.bits_of(o2), ref["out"], "foreign matrix scales")

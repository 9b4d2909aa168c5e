"""GPU parity of the tcgen05 expert-FFN kernel (forced), against the CPU oracle.

Covers token tiles of 32..256 columns, ragged expert row counts, split K (few tiles) and
whole layers; every call's workspace error word (bounded waits inside the kernel) must be 0.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import bf16, moe_ref

from gpu_util import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import expert_dispatch_streaming_gb300 as m
    m.set_ffn_kernel("tcgen05")
    m.set_decode_kernel(False)          # small batches too run the step-by-step kernels here
    yield m
    m.set_decode_kernel(True)
    m.set_ffn_kernel("auto")


@pytest.fixture(scope="module")
def syn(moe):
    from expert_dispatch_streaming_gb300 import synthetic
    return synthetic


def _grouped(moe, syn, cfg, counts, seed=0):
    """Run moe_grouped_swiglu on random x rows grouped by the given per-expert counts."""
    rng = np.random.default_rng(seed)
    rows = int(sum(counts))
    xb = wl.bf16_bits_from_f32(rng.standard_normal((rows, cfg.H)).astype(np.float32))
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    dl = syn.DeviceLayer(cfg)
    y = torch.zeros((rows, cfg.H), dtype=torch.int16, device="cuda")
    nws = moe.moe_grouped_swiglu_workspace_size(rows, cfg.E, cfg.H, cfg.I, cfg.wdtype)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    moe.moe_grouped_swiglu(syn.to_device_bits(xb), torch.from_numpy(offsets).cuda(),
                           [dl.routed[e] for e in range(cfg.E)], cfg.E, cfg.H, cfg.I, cfg.wdtype,
                           rows, y, ws, nws)
    torch.cuda.synchronize()
    assert moe.moe_workspace_error(ws) == 0
    got = y.cpu().numpy().view(np.uint16)
    x = bf16.decode(xb)
    ref = np.zeros((rows, cfg.H))
    for e in range(cfg.E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            wg, wu, wd = moe_ref.expert_matrices(wl.expert(cfg, 0, e))
            ref[lo:hi], _ = moe_ref.swiglu_ffn(x[lo:hi], wg, wu, wd)
    return got, ref


@pytest.mark.parametrize("counts", [
    [1, 0, 3, 0, 0, 2, 0, 1],          # decode-like: BN 32, split K
    [40, 7, 0, 33, 64, 1, 0, 90],      # ragged, BN 64
    [300, 5, 129, 0, 0, 0, 0, 256],    # BN 128/256, several token tiles per expert
])
def test_grouped_tcgen05_bf16(moe, syn, counts):
    cfg = wl.custom("tc", cfg_id=120, H=512, E=8, k=2, I=384)
    got, ref = _grouped(moe, syn, cfg, counts)
    assert_close(got, ref, f"tcgen05 counts={counts}")


@pytest.mark.parametrize("wdtype", ["int4_g128", "nvfp4"])
def test_grouped_tcgen05_quantised_wide_token_tiles(moe, syn, wdtype):
    """Quantised weights take 128-token tiles here (the grouped call bounds no expert's rows
    below the batch): experts with 1, 5, 33 and 70 rows load only their 32-row boxes, and
    300 / 129 rows span several tiles with ragged ends."""
    cfg = wl.custom("tcq_" + wdtype, cfg_id=123, H=512, E=8, k=2, I=384, wdtype=wdtype)
    got, ref = _grouped(moe, syn, cfg, [300, 5, 129, 0, 33, 1, 0, 70])
    assert_close(got, ref, f"tcgen05 {wdtype} wide token tiles")


def test_grouped_tcgen05_large_k(moe, syn):
    cfg = wl.custom("tck", cfg_id=121, H=2048, E=4, k=2, I=1408)
    got, ref = _grouped(moe, syn, cfg, [600, 3, 0, 257])
    assert_close(got, ref, "tcgen05 H=2048 I=1408")


@pytest.mark.parametrize("T", [1, 64, 700])
def test_layer_tcgen05_qwen_shape(moe, syn, T):
    cfg = wl.QWEN
    dl = syn.DeviceLayer(cfg)
    xb = wl.tokens(cfg, T)
    x = syn.to_device_bits(xb)
    ws = dl.workspace(T)
    ids = torch.empty((T, cfg.k), dtype=torch.int32, device="cuda")
    out, _ = dl.forward(x, ws, ids_out=ids)
    torch.cuda.synchronize()
    assert moe.moe_workspace_error(ws) == 0
    rows = np.arange(T) if T <= 64 else np.arange(0, T, 37)
    ref = moe_ref.layer_forward(cfg, 0, xb, forced_ids=ids.cpu().numpy(), rows=rows)
    assert_close(syn.bits_of(out)[rows], ref["out"], f"qwen T={T} tcgen05")


def test_layer_tcgen05_mixtral_prefill_sampled(moe, syn):
    cfg = wl.MIXTRAL
    T = 4096
    dl = syn.DeviceLayer(cfg)
    xb = wl.tokens(cfg, T)
    x = syn.to_device_bits(xb)
    ws = dl.workspace(T)
    ids = torch.empty((T, cfg.k), dtype=torch.int32, device="cuda")
    out, _ = dl.forward(x, ws, ids_out=ids)
    out2, _ = dl.forward(x, ws)
    torch.cuda.synchronize()
    assert moe.moe_workspace_error(ws) == 0
    got = syn.bits_of(out)
    assert np.array_equal(got, syn.bits_of(out2))
    rows = np.array([0, 1, 777, 2048, 4095])
    ref = moe_ref.layer_forward(cfg, 0, xb, forced_ids=ids.cpu().numpy(), rows=rows)
    assert_close(got[rows], ref["out"], "mixtral T=4096 tcgen05 sampled rows")


@pytest.mark.parametrize("T", [1, 40, 300])
def test_layer_tcgen05_int4_with_shared_expert(moe, syn, T):
    """INT4 routed + shared expert in one tcgen05 launch per GEMM (split K at small T)."""
    cfg = wl.custom("ds_tc", cfg_id=122, H=512, E=64, k=8, I=256, gating="sigmoid_bias_renorm",
                    scale=2.5, Is=384, shared_gate="one", wdtype="int4_g128", zipf_s=1.1,
                    bias_kind="select")
    dl = syn.DeviceLayer(cfg)
    xb = wl.tokens(cfg, T)
    x = syn.to_device_bits(xb)
    ws = dl.workspace(T)
    ids = torch.empty((T, cfg.k), dtype=torch.int32, device="cuda")
    out, _ = dl.forward(x, ws, ids_out=ids)
    torch.cuda.synchronize()
    assert moe.moe_workspace_error(ws) == 0
    ref = moe_ref.layer_forward(cfg, 0, xb, forced_ids=ids.cpu().numpy())
    assert_close(syn.bits_of(out), ref["out"], f"int4 + shared T={T} tcgen05")


@pytest.mark.parametrize("name,T", [("qwen", 1), ("qwen", 16), ("qwen", 700), ("ds", 40)])
def test_layer_bits_identical_with_and_without_programmatic_launch(moe, syn, name, T):
    """Programmatic dependent launch only moves when kernels are scheduled: every kernel waits
    for its predecessor's results in-kernel, so the outputs are bit-identical to plain launches
    (a missing wait would show up here as a race)."""
    cfg = wl.QWEN if name == "qwen" else wl.custom(
        "ds_pdl", cfg_id=123, H=512, E=64, k=8, I=256, gating="sigmoid_bias_renorm", scale=2.5,
        Is=384, shared_gate="one", wdtype="int4_g128", zipf_s=1.1, bias_kind="select")
    dl = syn.DeviceLayer(cfg)
    xb = wl.tokens(cfg, T)
    x = syn.to_device_bits(xb)
    ws = dl.workspace(T)
    outs = []
    try:
        for pdl in (True, False, True):
            moe.set_pdl(pdl)
            out, _ = dl.forward(x, ws)
            out2, _ = dl.forward(out, ws)        # a second layer call fed by the first
            torch.cuda.synchronize()
            assert moe.moe_workspace_error(ws) == 0
            outs.append((syn.bits_of(out), syn.bits_of(out2)))
    finally:
        moe.set_pdl(False)
    for a, b in outs[1:]:
        assert np.array_equal(a, outs[0][0]) and np.array_equal(b, outs[0][1])

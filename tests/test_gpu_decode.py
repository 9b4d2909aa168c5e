"""GPU parity of the fused decode kernel (a batch of at most 16 tokens with every bundle
resident runs as one cooperative launch) against the CPU oracle and the step-by-step path.

Routing ids bit-exact (except logged near-ties), outputs within max |err| <= 2e-2 max |ref| and
sum |err| / sum |ref| <= 5e-3; the pre-normalised stack's RMS output within one bf16 step.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import bf16, moe_ref

from gpu_util import assert_close, check_ids

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import expert_dispatch_streaming_gb300 as m
    m.set_decode_kernel("always")
    yield m
    m.set_decode_kernel("auto")


@pytest.fixture(scope="module")
def syn(moe):
    from expert_dispatch_streaming_gb300 import synthetic
    return synthetic


SMALL = [
    wl.TINY,
    wl.custom("dec_qwen", cfg_id=170, H=512, E=60, k=4, I=384, gating="softmax", Is=640,
              shared_gate="sigmoid", zipf_s=1.0, bias_kind="logit"),
    wl.custom("dec_ds", cfg_id=171, H=768, E=64, k=8, I=256, gating="sigmoid_bias_renorm",
              scale=2.5, Is=256, shared_gate="one", wdtype="int4_g128", zipf_s=1.1,
              bias_kind="select"),
    wl.custom("dec_fp4", cfg_id=172, H=384, E=16, k=4, I=512, gating="softmax", Is=256,
              shared_gate="sigmoid", zipf_s=1.0, bias_kind="logit", wdtype="nvfp4"),
    wl.custom("dec_big_i", cfg_id=173, H=256, E=8, k=2, I=1024, gating="softmax_renorm"),
]


def _run(moe, syn, dl, cfg, xb, T, residual=None, normed=False, forced=None, decode=True):
    moe.set_decode_kernel("always" if decode else "off")
    try:
        x = syn.to_device_bits(xb)
        ws = dl.workspace(T)
        ids = torch.empty((T, cfg.k), dtype=torch.int32, device="cuda")
        res = syn.to_device_bits(residual) if residual is not None else None
        un = torch.empty_like(x) if normed else None
        f = torch.from_numpy(np.ascontiguousarray(forced, np.int32)).cuda() if forced is not None else None
        out, st = dl.forward(x, ws, ids_out=ids, residual=res, out_normed=un, forced_ids=f)
        torch.cuda.synchronize()
        assert moe.moe_workspace_error(ws) == 0
        return (syn.bits_of(out), ids.cpu().numpy(), syn.bits_of(un) if normed else None, st)
    finally:
        moe.set_decode_kernel("always")


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
@pytest.mark.parametrize("T", [1, 2, 5, 8, 9, 16])
def test_decode_kernel_matches_oracle(moe, syn, cfg, T):
    dl = syn.DeviceLayer(cfg)
    xb = wl.tokens(cfg, T)
    out, ids, _, st = _run(moe, syn, dl, cfg, xb, T)
    assert st.fused_decode == 1 and st.n_launches == 1
    check_ids(cfg, ids, None, xb)
    ref = moe_ref.layer_forward(cfg, 0, xb, forced_ids=ids)
    assert_close(out, ref["out"], f"{cfg.name} T={T}")
    # deterministic: a second call gives the same bits
    out2, ids2, _, _ = _run(moe, syn, dl, cfg, xb, T)
    assert np.array_equal(out, out2) and np.array_equal(ids, ids2)


@pytest.mark.parametrize("cfg", SMALL[1:4], ids=lambda c: c.name)
def test_decode_kernel_against_step_by_step_path(moe, syn, cfg):
    """Same ids, and outputs within the tolerance of each other (the sums run in a different
    fixed order), with a residual and the RMS-normalised output."""
    T = 11
    dl = syn.DeviceLayer(cfg)
    xb = wl.tokens(cfg, T)
    resb = wl.tokens(cfg, T, step=3)
    a_out, a_ids, a_n, _ = _run(moe, syn, dl, cfg, xb, T, residual=resb, normed=True)
    b_out, b_ids, b_n, st = _run(moe, syn, dl, cfg, xb, T, residual=resb, normed=True,
                                 decode=False)
    assert st.fused_decode == 0
    assert np.array_equal(a_ids, b_ids)
    ref = bf16.round_rne(bf16.decode(resb)
                         + moe_ref.layer_forward(cfg, 0, xb, forced_ids=a_ids)["out"])
    assert_close(a_out, ref, "decode + residual")
    assert_close(b_out, ref, "step-by-step + residual")
    refn = moe_ref.rms_normalize(bf16.decode(a_out), wl.STACK_NORM_EPS)
    gotn = bf16.decode(a_n)
    assert np.abs(gotn - refn).max() <= 2 ** -7 * np.abs(refn).max()


def test_decode_kernel_forced_ids(moe, syn):
    cfg = SMALL[1]
    T = 7
    rng = np.random.default_rng(11)
    forced = np.stack([rng.choice(cfg.E, cfg.k, replace=False) for _ in range(T)]).astype(np.int32)
    dl = syn.DeviceLayer(cfg)
    xb = wl.tokens(cfg, T)
    out, ids, _, _ = _run(moe, syn, dl, cfg, xb, T, forced=forced)
    assert np.array_equal(ids, forced)
    assert_close(out, moe_ref.layer_forward(cfg, 0, xb, forced_ids=forced)["out"], "forced")


@pytest.mark.parametrize("name,T", [("mixtral", 1), ("mixtral", 8), ("qwen", 1), ("qwen", 16),
                                    ("deepseek", 1), ("deepseek", 16), ("qwen_nvfp4", 1),
                                    ("qwen_nvfp4", 16)])
def test_decode_kernel_full_shapes(moe, syn, name, T):
    cfg = {"mixtral": wl.MIXTRAL, "qwen": wl.QWEN, "deepseek": wl.DEEPSEEK,
           "qwen_nvfp4": wl.QWEN_NVFP4}[name]
    dl = syn.DeviceLayer(cfg)
    xb = wl.tokens(cfg, T)
    out, ids, _, st = _run(moe, syn, dl, cfg, xb, T)
    assert st.fused_decode == 1
    check_ids(cfg, ids, None, xb)
    ref = moe_ref.layer_forward(cfg, 0, xb, forced_ids=ids)
    assert_close(out, ref["out"], f"{name} T={T}")


def test_decode_kernel_replays_as_a_cuda_graph(moe, syn):
    cfg = SMALL[2]
    T = 4
    dl = syn.DeviceLayer(cfg)
    x = syn.to_device_bits(wl.tokens(cfg, T))
    ws = dl.workspace(T)
    out = torch.empty_like(x)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        dl.forward(x, ws, out=out, stream=stream)
    stream.synchronize()
    eager = syn.bits_of(out).copy()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        dl.forward(x, ws, out=out, stream=stream)
    out.zero_()
    for _ in range(3):
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        assert np.array_equal(syn.bits_of(out), eager)
    assert moe.moe_workspace_error(ws) == 0

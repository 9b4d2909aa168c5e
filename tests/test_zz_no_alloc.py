"""The allocation-free routing entry point (moe_route_topk_static) against moe_route_topk.

Some callers cannot allocate device memory (a plug-in inside a framework that owns all device
memory, or a latency-critical path that must not call cudaMalloc / cudaFree), so the library
offers one routing call whose scratch is a fixed array in its own device memory.  This test
calls it through the C ABI twice in a row -- the second call sees the array as the first one
left it -- and checks both results against the workspace-based call, plus the size limit.
Collected last on purpose: a failure here does not stop the rest of the suite.
"""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import expert_dispatch_streaming_gb300 as m
    return m


def _inputs(cfg, T):
    from expert_dispatch_streaming_gb300.synthetic import to_device_bits
    dev = "cuda"
    x = to_device_bits(wl.tokens(cfg, T))
    w_r = torch.from_numpy(wl.router(cfg, 0)).to(dev)
    b = wl.popularity_bias(cfg, 0)
    lb = torch.from_numpy(b).to(dev) if (b is not None and cfg.bias_kind == "logit") else None
    sb = torch.from_numpy(b).to(dev) if (b is not None and cfg.bias_kind == "select") else None
    wsv = wl.shared_gate_vector(cfg, 0)
    wg = to_device_bits(wsv) if wsv is not None else None
    return x, w_r, lb, sb, wg


def _outputs(cfg, T):
    i32 = dict(dtype=torch.int32, device="cuda")
    return dict(ids=torch.full((T, cfg.k), -1, **i32),
                w=torch.zeros((T, cfg.k), dtype=torch.float32, device="cuda"),
                counts=torch.full((cfg.E,), -1, **i32), offsets=torch.full((cfg.E + 1,), -1, **i32),
                pos=torch.full((T, cfg.k), -1, **i32), src=torch.full((T * cfg.k,), -1, **i32),
                logits=torch.zeros((T, cfg.E), dtype=torch.float32, device="cuda"),
                sg=torch.zeros(T, dtype=torch.float32, device="cuda"),
                tie=torch.full((T,), -1, **i32))


CASES = [
    (wl.custom("na_qwen", cfg_id=140, H=512, E=60, k=4, I=256, gating="softmax", Is=256,
               shared_gate="sigmoid", zipf_s=1.0, bias_kind="logit"), 37),
    (wl.custom("na_ds", cfg_id=141, H=1024, E=256, k=8, I=256, gating="sigmoid_bias_renorm",
               scale=2.5, zipf_s=1.1, bias_kind="select"), 300),
    (wl.TINY, 16),
]


@pytest.mark.parametrize("cfg,T", CASES, ids=lambda v: getattr(v, "name", str(v)))
def test_static_scratch_matches_workspace_call(moe, cfg, T):
    x, w_r, lb, sb, wg = _inputs(cfg, T)
    ref = _outputs(cfg, T)
    nws = moe.moe_route_workspace_size(T, cfg.H, cfg.E, cfg.k)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    sg_ref = ref["sg"] if wg is not None else None
    moe.moe_route_topk(x, w_r, lb, sb, wg, None, T, cfg.H, cfg.E, cfg.k, cfg.gating, cfg.scale,
                       ref["ids"], ref["w"], ref["counts"], ref["offsets"], ref["pos"], ref["src"],
                       ref["logits"], sg_ref, ref["tie"], ws, nws)
    for _ in range(2):                      # two calls in a row share the static array
        got = _outputs(cfg, T)
        sg_got = got["sg"] if wg is not None else None
        moe.moe_route_topk_static(x, w_r, lb, sb, wg, None, T, cfg.H, cfg.E, cfg.k, cfg.gating,
                                  cfg.scale, got["ids"], got["w"], got["counts"], got["offsets"],
                                  got["pos"], got["src"], got["logits"], sg_got, got["tie"])
        torch.cuda.synchronize()
        for key in ("ids", "counts", "offsets", "pos", "src", "tie"):
            assert torch.equal(got[key].cpu(), ref[key].cpu()), key
        assert torch.allclose(got["w"], ref["w"], rtol=0, atol=1e-6)
        assert torch.allclose(got["logits"], ref["logits"], rtol=0, atol=1e-5)
        if wg is not None:
            assert torch.allclose(got["sg"], ref["sg"], rtol=0, atol=1e-6)
        # the fixed array's error word (bounded waits of the tensor-core router) reads clean
        assert moe.moe_route_static_error() == 0


def test_static_scratch_rejects_oversized_request(moe):
    T, H, E, k = 8192, 7168, 256, 8          # needs more than the fixed 8 MiB of scratch
    assert moe.moe_route_workspace_size(T, H, E, k) > (8 << 20)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_route_topk_static(1, 1, None, None, None, None, T, H, E, k, 2, 2.5, 1, 1, 1, 1,
                                  1, 1, None, None, None)
    assert ei.value.status == moe.MOE_ERR_CAPACITY

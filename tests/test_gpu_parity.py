"""GPU parity: every step of the MoE layer, called through the C ABI, against the CPU oracle.

Bit-exact: routing ids (except near-ties), counts, offsets, pos, src, the permuted rows.
Tolerance (floating point): max |err| <= 2e-2 max |ref|, sum |err| / sum |ref| <= 5e-3.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import bf16, moe_ref

from gpu_util import assert_close, check_ids, oracle_scores, spread_rows

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
    wl.TINY,
    wl.custom("ragged", H=256, E=8, k=2, I=384),
    wl.custom("qwenlike", cfg_id=101, H=512, E=60, k=4, I=256, gating="softmax", Is=384,
              shared_gate="sigmoid", zipf_s=1.0, bias_kind="logit"),
    wl.custom("dslike", cfg_id=102, H=512, E=256, k=8, I=256, gating="sigmoid_bias_renorm",
              scale=2.5, Is=256, shared_gate="one", wdtype="int4_g128", zipf_s=1.1,
              bias_kind="select"),
    wl.custom("int4small", cfg_id=103, H=256, E=16, k=4, I=384, gating="softmax_renorm",
              wdtype="int4_g128"),
]


def _route(moe, cfg, T, forced=None, w_r=None, logit_bias=None):
    dev = "cuda"
    from expert_dispatch_streaming_gb300.synthetic import to_device_bits
    xb = wl.tokens(cfg, T)
    x = to_device_bits(xb)
    w_r = torch.from_numpy(wl.router(cfg, 0) if w_r is None else w_r).to(dev)
    b = wl.popularity_bias(cfg, 0) if logit_bias is None else logit_bias
    lb = torch.from_numpy(b).to(dev) if (b is not None and (cfg.bias_kind == "logit" or logit_bias is not None)) else None
    sb = torch.from_numpy(b).to(dev) if (b is not None and cfg.bias_kind == "select") else None
    wsv = wl.shared_gate_vector(cfg, 0)
    wg = to_device_bits(wsv) if wsv is not None else None
    E, k = cfg.E, cfg.k
    i32 = dict(dtype=torch.int32, device=dev)
    ids = torch.full((T, k), -1, **i32)
    w = torch.zeros((T, k), dtype=torch.float32, device=dev)
    counts = torch.zeros(E, **i32)
    offsets = torch.zeros(E + 1, **i32)
    pos = torch.full((T, k), -1, **i32)
    src = torch.full((T * k,), -1, **i32)
    logits = torch.zeros((T, E), dtype=torch.float32, device=dev)
    sg = torch.zeros(T, dtype=torch.float32, device=dev) if wg is not None else None
    tie = torch.zeros(T, **i32)
    nws = moe.moe_route_workspace_size(T, cfg.H, E, k)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    f = torch.from_numpy(np.ascontiguousarray(forced, np.int32)).to(dev) if forced is not None else None
    moe.moe_route_topk(x, w_r, lb, sb, wg, f, T, cfg.H, E, k, cfg.gating, cfg.scale, ids, w,
                       counts, offsets, pos, src, logits, sg, tie, ws, nws)
    torch.cuda.synchronize()
    out = dict(ids=ids.cpu().numpy(), w=w.cpu().numpy(), counts=counts.cpu().numpy(),
               offsets=offsets.cpu().numpy(), pos=pos.cpu().numpy(), src=src.cpu().numpy(),
               logits=logits.cpu().numpy(), tie=tie.cpu().numpy(),
               sg=sg.cpu().numpy() if sg is not None else None)
    return xb, out


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
@pytest.mark.parametrize("T", [1, 3, 17, 130, 300])
def test_route_topk_dispatch(moe, cfg, T):
    xb, g = _route(moe, cfg, T)
    l, s = oracle_scores(cfg, xb)
    assert np.abs(g["logits"] - l).max() < 1e-3
    check_ids(cfg, g["ids"], g["tie"], xb)
    # second stage: dispatch of the GPU's own ids must match the definition bit for bit
    counts, offsets, pos, src = moe_ref.dispatch(g["ids"], cfg.E)
    assert np.array_equal(g["counts"], counts) and np.array_equal(g["offsets"], offsets)
    assert np.array_equal(g["pos"], pos) and np.array_equal(g["src"], src)
    w_ref = moe_ref.gate_weights(l, g["ids"], cfg.gating, cfg.scale)
    assert np.abs(g["w"] - w_ref).max() <= 1e-5 * max(1.0, cfg.scale)
    if g["sg"] is not None:
        x = bf16.decode(xb)
        ref = moe_ref.sigmoid(x @ bf16.decode(wl.shared_gate_vector(cfg, 0)))
        assert np.abs(g["sg"] - ref).max() < 1e-5


@pytest.mark.parametrize("cfg,T", [(wl.DEEPSEEK, 2048), (wl.QWEN, 4096), (wl.MIXTRAL, 1024)],
                         ids=["deepseek-2048", "qwen-4096", "mixtral-1024"])
def test_route_tensor_core_router_full_shapes(moe, cfg, T):
    """Batches of >= 256 tokens compute the router product on the tensor cores (bf16 x 3
    pieces); selection must still equal exact arithmetic away from near-ties."""
    xb, g = _route(moe, cfg, T)
    l, s = oracle_scores(cfg, xb)
    assert np.abs(g["logits"] - l).max() < 1e-3
    n_near = check_ids(cfg, g["ids"], g["tie"], xb)
    counts, offsets, pos, src = moe_ref.dispatch(g["ids"], cfg.E)
    assert np.array_equal(g["pos"], pos) and np.array_equal(g["src"], src)
    assert n_near <= max(2, T // 500)


def test_route_forced_ids(moe):
    cfg = SMALL[2]
    T = 37
    rng = np.random.default_rng(5)
    forced = np.stack([rng.choice(cfg.E, cfg.k, replace=False) for _ in range(T)]).astype(np.int32)
    xb, g = _route(moe, cfg, T, forced=forced)
    assert np.array_equal(g["ids"], forced)
    l, _ = oracle_scores(cfg, xb)
    assert np.abs(g["w"] - moe_ref.gate_weights(l, forced, cfg.gating, cfg.scale)).max() < 1e-5
    counts, offsets, pos, src = moe_ref.dispatch(forced, cfg.E)
    assert np.array_equal(g["pos"], pos) and np.array_equal(g["src"], src)


def test_route_near_tie_refinement(moe):
    # experts 1 and 2 have identical router columns and biases, expert 5 a bias far above
    # everything: every token's k-th (2nd) place is an exact tie between 1 and 2, so every
    # token must go through fp64 re-scoring, be logged as a near-tie and take the lower id
    cfg = wl.custom("ties", H=256, E=8, k=2, I=128)
    w = wl.router(cfg, 0).copy()
    w[:, 2] = w[:, 1]
    bias = np.zeros(cfg.E, np.float32)
    bias[5], bias[1], bias[2] = 20.0, 10.0, 10.0
    xb, g = _route(moe, cfg, 40, w_r=w, logit_bias=bias)
    assert np.all(g["tie"] == 2)
    assert np.all(g["ids"][:, 0] == 1) and np.all(g["ids"][:, 1] == 5)   # ascending ids


@pytest.mark.parametrize("T,k,H", [(1, 2, 256), (37, 4, 512), (300, 8, 7168)])
def test_permute_bit_exact(moe, T, k, H):
    rng = np.random.default_rng(T)
    x = torch.from_numpy(rng.integers(-32768, 32767, (T, H), dtype=np.int16)).cuda()
    src = torch.from_numpy(rng.permutation(T * k).astype(np.int32)).cuda()
    out = torch.empty((T * k, H), dtype=torch.int16, device="cuda")
    moe.moe_permute(x, src, T, k, H, out)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), x.cpu()[src.cpu().long() // k])


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_grouped_swiglu(moe, syn, cfg):
    T = 57
    xb, g = _route(moe, cfg, T)
    x = bf16.decode(xb)
    rows = T * cfg.k
    x_perm = torch.from_numpy(xb.view(np.int16)[g["src"] // cfg.k].copy()).cuda()
    offsets = torch.from_numpy(g["offsets"]).cuda()
    dl = syn.DeviceLayer(cfg)
    y = torch.zeros((rows, cfg.H), dtype=torch.int16, device="cuda")
    nws = moe.moe_grouped_swiglu_workspace_size(rows, cfg.E, cfg.H, cfg.I, cfg.wdtype)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    moe.moe_grouped_swiglu(x_perm, offsets, [dl.routed[e] for e in range(cfg.E)], cfg.E, cfg.H,
                           cfg.I, cfg.wdtype, rows, y, ws, nws)
    torch.cuda.synchronize()
    y = y.cpu().numpy().view(np.uint16)
    ref = np.zeros((rows, cfg.H))
    for e in range(cfg.E):
        lo, hi = g["offsets"][e], g["offsets"][e + 1]
        if hi > lo:
            wg, wu, wd = moe_ref.expert_matrices(wl.expert(cfg, 0, e))
            ref[lo:hi], _ = moe_ref.swiglu_ffn(x[g["src"][lo:hi] // cfg.k], wg, wu, wd)
    assert_close(y, ref, f"{cfg.name} y_perm")


def test_combine(moe):
    rng = np.random.default_rng(3)
    T, k, H = 77, 4, 512
    y = wl.bf16_bits_from_f32(rng.standard_normal((T * k, H)).astype(np.float32))
    s = wl.bf16_bits_from_f32(rng.standard_normal((T, H)).astype(np.float32))
    res = wl.bf16_bits_from_f32(rng.standard_normal((T, H)).astype(np.float32))
    pos = rng.permutation(T * k).astype(np.int32).reshape(T, k)
    w = rng.random((T, k)).astype(np.float32)
    gate = rng.random(T).astype(np.float32)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else a).cuda()  # noqa
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    out2 = torch.empty((T, H), dtype=torch.int16, device="cuda")
    moe.moe_combine(d(y), d(pos), d(w), T, k, H, d(s), d(gate), None, out)
    moe.moe_combine(d(y), d(pos), d(w), T, k, H, d(s), d(gate), d(res), out2)
    torch.cuda.synchronize()
    ref = moe_ref.combine(bf16.decode(y), pos, w.astype(np.float64), bf16.decode(s),
                          gate.astype(np.float64))
    got = out.cpu().numpy().view(np.uint16)
    assert_close(got, ref, "combine")
    # fp32 accumulation vs fp64: at most one bf16 step apart
    assert np.mean(bf16.decode(got) == ref) > 0.98
    ref2 = bf16.round_rne(bf16.decode(res) + ref)
    assert_close(out2.cpu().numpy().view(np.uint16), ref2, "combine+residual")
    # the RMS-normalised output of a pre-norm stack, from the bf16 values of out itself
    for H2 in (H, 7168):
        y2 = wl.bf16_bits_from_f32(rng.standard_normal((T * k, H2)).astype(np.float32))
        r2 = wl.bf16_bits_from_f32(rng.standard_normal((T, H2)).astype(np.float32))
        o3 = torch.empty((T, H2), dtype=torch.int16, device="cuda")
        n3 = torch.empty((T, H2), dtype=torch.int16, device="cuda")
        moe.moe_combine(d(y2), d(pos), d(w), T, k, H2, None, None, d(r2), o3, out_normed=n3,
                        norm_eps=1e-6)
        torch.cuda.synchronize()
        got3 = o3.cpu().numpy().view(np.uint16)
        ref3 = bf16.round_rne(bf16.decode(r2) + moe_ref.combine(bf16.decode(y2), pos,
                                                                w.astype(np.float64)))
        assert_close(got3, ref3, f"combine+residual H={H2}")
        refn = moe_ref.rms_normalize(bf16.decode(got3), 1e-6)
        gotn = bf16.decode(n3.cpu().numpy().view(np.uint16))
        assert_close(n3.cpu().numpy().view(np.uint16), refn, f"normalised H={H2}")
        assert np.abs(gotn - refn).max() <= 2 ** -7 * np.abs(refn).max()   # one bf16 step
        assert np.mean(gotn == refn) > 0.98


def _layer_case(syn, cfg, T, rows=None, check_selection=True):
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
    if check_selection:
        check_ids(cfg, ids, None, xb)
    if isinstance(rows, str) and rows == "spread":
        rows = spread_rows(ids, cfg.E)
    ref = moe_ref.layer_forward(cfg, 0, xb, forced_ids=ids, rows=rows)
    sel = ref["rows"]
    return assert_close(got[sel], ref["out"], f"{cfg.name} T={T}")


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
@pytest.mark.parametrize("T", [1, 16, 133])
def test_layer_forward_small(syn, cfg, T):
    _layer_case(syn, cfg, T)


@pytest.mark.parametrize("T", [1, 8, 64])
def test_layer_forward_mixtral(syn, T):
    _layer_case(syn, wl.MIXTRAL, T)


@pytest.mark.parametrize("T", [1, 16, 256])
def test_layer_forward_qwen(syn, T):
    _layer_case(syn, wl.QWEN, T)


@pytest.mark.parametrize("T", [1, 32, 512, 8192])
def test_layer_forward_deepseek_int4(syn, T):
    """The DeepSeek-V3-shaped INT4 layer (256 experts, top-8 sigmoid, shared expert) at every
    batch size of the workload; rows spread over the batch (incl. the last token of the busiest
    experts, whose ragged last token tile the first rows never reach)."""
    _layer_case(syn, wl.DEEPSEEK, T, rows="spread")


@pytest.mark.parametrize("T", [2048, 8192])
def test_layer_forward_qwen_large(syn, T):
    """The Qwen1.5-MoE-shaped layer (60 experts, shared expert) at the large batch sizes of
    the workload, on rows spread over the batch."""
    _layer_case(syn, wl.QWEN, T, rows="spread")


def test_int4_bundle_with_foreign_scales_fails_parity(moe, syn):
    """Scales travel with their weights: a bundle whose scale block comes from another expert
    gives a wrong layer (the negative test of bundle atomicity)."""
    cfg = SMALL[4]
    hb = syn.host_bundles(cfg, 0, list(range(cfg.E)), pinned=False)
    lay = moe.bundle_layout(cfg.H, cfg.I, cfg.wdtype)
    bad = hb.clone()
    tiles = [lay.gate_up_offset + t * 8448 for t in range((2 * cfg.I // 128) * (cfg.H // 128))]
    tiles += [lay.down_offset + t * 8448 for t in range((cfg.H // 128) * (cfg.I // 128))]
    for e in range(cfg.E):                      # only the scale block of every tile is foreign
        for t0 in tiles:
            bad[e, t0 + 8192:t0 + 8448] = hb[(e + 1) % cfg.E, t0 + 8192:t0 + 8448]
    T = 33
    xb = wl.tokens(cfg, T)
    x = syn.to_device_bits(xb)
    good_l, bad_l = syn.DeviceLayer(cfg, bundles_override=hb), syn.DeviceLayer(cfg, bundles_override=bad)
    ws = good_l.workspace(T)
    ids = torch.empty((T, cfg.k), dtype=torch.int32, device="cuda")
    o1, _ = good_l.forward(x, ws, ids_out=ids)
    o2, _ = bad_l.forward(x, ws)
    torch.cuda.synchronize()
    ref = moe_ref.layer_forward(cfg, 0, xb, forced_ids=ids.cpu().numpy())
    assert_close(syn.bits_of(o1), ref["out"], "good bundles")
    with pytest.raises(AssertionError):
        assert_close(syn.bits_of(o2), ref["out"], "foreign scales")


@pytest.mark.parametrize("cfg", [SMALL[1], SMALL[3], SMALL[4]], ids=lambda c: c.name)
@pytest.mark.parametrize("T", [1, 133])
def test_layer_forward_streaming_kernel(moe, syn, cfg, T):
    """The mma.sync weight-streaming FFN kernel (forced), bf16 and INT4."""
    moe.set_ffn_kernel("stream")
    moe.set_decode_kernel(False)
    try:
        _layer_case(syn, cfg, T)
    finally:
        moe.set_decode_kernel(True)
        moe.set_ffn_kernel("auto")


def test_layer_forward_empty_batch(moe, syn):
    cfg = SMALL[2]
    dl = syn.DeviceLayer(cfg)
    x = torch.empty((0, cfg.H), dtype=torch.int16, device="cuda")
    out = torch.empty((0, cfg.H), dtype=torch.int16, device="cuda")
    ws = dl.workspace(1)
    st = moe.moe_layer_forward(dl.desc, x, 0, None, None, out, None, ws, ws.numel())
    assert st.n_launches == 0


def test_layer_k_equals_E_is_dense_mixture_on_gpu(syn):
    """Top-k with k = E (softmax renormalised over all) equals the dense gate-weighted mixture."""
    cfg = wl.custom("dense", cfg_id=150, H=256, E=8, k=8, I=256)
    _layer_case(syn, cfg, 37)
    xb = wl.tokens(cfg, 37)
    x = bf16.decode(xb)
    l = x @ wl.router(cfg, 0).astype(np.float64)
    gates = np.exp(l - l.max(1, keepdims=True))
    gates /= gates.sum(1, keepdims=True)
    experts = [moe_ref.expert_matrices(wl.expert(cfg, 0, e)) for e in range(cfg.E)]
    ref = moe_ref.dense_mixture(x, gates, experts)
    dl = syn.DeviceLayer(cfg)
    out, _ = dl.forward(syn.to_device_bits(xb), dl.workspace(37))
    torch.cuda.synchronize()
    assert_close(syn.bits_of(out), ref, "k = E vs dense mixture")


def test_layer_token_permutation_invariance_on_gpu(syn):
    """Permuting tokens permutes the outputs bit for bit (no cross-token arithmetic)."""
    cfg = SMALL[2]
    T = 300
    xb = wl.tokens(cfg, T)
    perm = np.random.default_rng(7).permutation(T)
    dl = syn.DeviceLayer(cfg)
    ws = dl.workspace(T)
    a, _ = dl.forward(syn.to_device_bits(xb), ws)
    a = syn.bits_of(a)
    b, _ = dl.forward(syn.to_device_bits(xb[perm]), ws)
    torch.cuda.synchronize()
    assert np.array_equal(a[perm], syn.bits_of(b))


def test_one_hot_router_on_gpu_reproduces_single_expert(moe, syn):
    """A router whose column e* beats every other logit by ~100 sends every token to e* with
    weight 1: the layer output is that expert's FFN (oracle SwiGLU of that expert)."""
    cfg = wl.custom("onehot", cfg_id=151, H=256, E=8, k=1, I=256)
    T, star = 21, 5
    x = bf16.decode(wl.tokens(cfg, T))
    s = x.sum(1)
    x = bf16.round_rne(x * (100.0 / np.where(np.abs(s) < 1e-3, 1e-3, s))[:, None])
    w_r = np.zeros((cfg.H, cfg.E), np.float32)
    w_r[:, star] = 1.0
    dl = syn.DeviceLayer(cfg)
    dl.w_r.copy_(torch.from_numpy(w_r))
    ids = torch.empty((T, 1), dtype=torch.int32, device="cuda")
    w = torch.empty((T, 1), dtype=torch.float32, device="cuda")
    out, _ = dl.forward(syn.to_device_bits(bf16.to_bits(x)), dl.workspace(T), ids_out=ids, w_out=w)
    torch.cuda.synchronize()
    assert np.all(ids.cpu().numpy() == star) and np.all(w.cpu().numpy() == 1.0)
    wg, wu, wd = moe_ref.expert_matrices(wl.expert(cfg, 0, star))
    y, _ = moe_ref.swiglu_ffn(x, wg, wu, wd)
    assert_close(syn.bits_of(out), y, "one-hot router")

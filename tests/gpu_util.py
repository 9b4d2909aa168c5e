"""Helpers of the GPU parity tests: run library steps on seeded inputs, compare with the oracle."""
import numpy as np
import torch

import workloads as wl
from oracle import bf16, moe_ref

# output tolerance: max |err| <= 2e-2 * max |ref| and sum |err| / sum |ref| <= 5e-3
MAX_REL = 2e-2
MEAN_REL = 5e-3


def out_errors(got_bits: np.ndarray, ref: np.ndarray):
    got = bf16.decode(got_bits)
    err = np.abs(got - ref)
    scale = max(np.abs(ref).max(), 1e-30)
    return err.max() / scale, err.sum() / max(np.abs(ref).sum(), 1e-30)


def assert_close(got_bits, ref, what=""):
    mx, mean = out_errors(got_bits, ref)
    assert mx <= MAX_REL and mean <= MEAN_REL, f"{what}: max_rel={mx:.3e} mean_rel={mean:.3e}"
    return mx, mean


def oracle_scores(cfg, x_bits, layer=0):
    x = bf16.decode(x_bits)
    b = wl.popularity_bias(cfg, layer)
    l = moe_ref.router_logits(x, wl.router(cfg, layer), b if cfg.bias_kind == "logit" else None)
    s = moe_ref.selection_scores(l, cfg.gating, b if cfg.bias_kind == "select" else None)
    return l, s


def check_ids(cfg, ids_gpu, tie_flags, x_bits, layer=0):
    """Bit-exact ids except logged near-ties (oracle k-th/(k+1)-th gap below 1e-6).

    Returns the number of near-tie tokens."""
    l, s = oracle_scores(cfg, x_bits, layer)
    ids_o, gap = moe_ref.topk_select(s, cfg.k)
    near = gap < 1e-6
    bad = np.where(~near & np.any(ids_gpu != ids_o, axis=1))[0]
    assert bad.size == 0, (f"ids differ at tokens {bad[:8]} (gaps {gap[bad[:8]]}, "
                           f"flags {tie_flags[bad[:8]] if tie_flags is not None else None})")
    # near-tie tokens: the GPU's set must still be a valid top-k within the tie
    for t in np.where(near)[0]:
        chosen = s[t, ids_gpu[t]]
        rest = np.delete(s[t], ids_gpu[t])
        assert len(set(ids_gpu[t].tolist())) == cfg.k
        assert chosen.min() >= rest.max() - 1e-6
    return int(near.sum())


def spread_rows(ids: np.ndarray, E: int, n_random: int = 3, seed: int = 0) -> np.ndarray:
    """Token rows to compare at a full shape, spread over the batch: the first, middle and last
    token (the shared expert's group is every token), the first, middle and last token of the
    two busiest experts (their later and ragged last token tiles) and a few random tokens."""
    T, k = ids.shape
    counts = np.bincount(ids.reshape(-1), minlength=E)
    rows = {0, T // 2, T - 1}
    for e in np.argsort(-counts, kind="stable")[:2]:
        toks = np.where(np.any(ids == e, axis=1))[0]      # ascending: its rows in expert order
        if toks.size:
            rows |= {int(toks[0]), int(toks[toks.size // 2]), int(toks[-1])}
    rng = np.random.default_rng(seed)
    rows |= set(rng.integers(0, T, n_random).tolist())
    return np.array(sorted(rows))


# ------------------------------------------------------------------ stacked layers
# A stack is pre-normalised: layer l takes u_l and adds its output to the residual stream,
#   x_{l+1} = bf16(x_l + layer_l(u_l)),  u_0 = x_0,  u_{l+1} = rmsnorm(x_{l+1})
# (the library's combine writes u_{l+1} beside x_{l+1}).


def stack_buffers(T, H, device="cuda"):
    return [torch.empty((T, H), dtype=torch.int16, device=device) for _ in range(4)]


def run_stack_step(layers, ws, x0, ids_of_layer, bufs, cache=None, stream=None):
    """One pass of x0 through every layer; returns the final residual stream tensor."""
    x = u = x0
    for l, layer in enumerate(layers):
        y, un = bufs[l & 1], bufs[2 + (l & 1)]
        layer.forward(u, ws, out=y, forced_ids=ids_of_layer(l), residual=x, cache=cache,
                      stream=stream, out_normed=un)
        x, u = y, un
    return x


def oracle_stack(cfg, trace, T, step, eps=wl.STACK_NORM_EPS):
    """The oracle's stacked layers at decode step `step` (same chaining), as fp64 values."""
    x = bf16.decode(wl.stream_tokens(cfg, T, step))
    u = x
    for l in range(cfg.layers):
        r = moe_ref.layer_forward(cfg, l, bf16.to_bits(u), forced_ids=trace[step, l])
        x = bf16.round_rne(x + r["out"])
        u = moe_ref.rms_normalize(x, eps)
    return x


def run_stack_step_recorded(syn, layers, ws, x0, ids_of_layer, bufs, cache=None):
    """As run_stack_step, but reads every layer's input and outputs back to the host:
    a list of (u_l, x_l, x_{l+1}, u_{l+1}) bf16 bit arrays, one per layer."""
    io = []
    x = u = x0
    for l, layer in enumerate(layers):
        y, un = bufs[l & 1], bufs[2 + (l & 1)]
        u_b, x_b = syn.bits_of(u).copy(), syn.bits_of(x).copy()
        layer.forward(u, ws, out=y, forced_ids=ids_of_layer(l), residual=x, cache=cache,
                      out_normed=un)
        io.append((u_b, x_b, syn.bits_of(y).copy(), syn.bits_of(un).copy()))
        x, u = y, un
    return io


def check_stack_layers(cfg, trace, step, io, eps=wl.STACK_NORM_EPS, what=""):
    """Two-stage parity of a stack, layer by layer on the GPU's own inputs: the oracle layer
    on u_l gives x_{l+1} = bf16(x_l + out_l) within the output tolerance, and u_{l+1} is the
    oracle's RMS normalisation of the GPU's x_{l+1} (one bf16 step at most).  Comparing each
    layer on its own input keeps the check independent of how rounding differences grow
    through the layers."""
    for l, (u_b, x_b, y_b, un_b) in enumerate(io):
        r = moe_ref.layer_forward(cfg, l, u_b, forced_ids=trace[step, l])
        ref = bf16.round_rne(bf16.decode(x_b) + r["out"])
        assert_close(y_b, ref, f"{what} layer {l} output")
        refn = moe_ref.rms_normalize(bf16.decode(y_b), eps)
        gotn = bf16.decode(un_b)
        assert np.abs(gotn - refn).max() <= 2 ** -7 * np.abs(refn).max(), f"{what} layer {l} norm"

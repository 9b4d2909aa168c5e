"""fp64 reference of the MoE layer forward (test infrastructure only).

Each function states the step it restates.  The pages are the five web pages on running MoE
models with expert-granular streaming and caching:

* "NovaLLM: Running Massive MoE Models Fully In-Memory" -- section "2. Why MoE Is a Natural
  Breakthrough Point" (the router picks a handful of experts per token and unselected experts
  are skipped) and "3. Optimization #1 -- Expert-Level Streaming" (per-expert storage; only
  the experts a batch hits need to be resident);
* "Running 35B MoE Models on 8GB GPUs: How vvllm-ms Caches Experts in System RAM" -- section
  "Technical Insight" (the cache sits between router output and expert computation; an expert
  bundle is weights plus quantisation scales and moves as one unit; LRU eviction).

The pages do not write out the MoE arithmetic.  The formulas below are the standard ones the
workload definitions name: softmax top-k renormalised over the chosen experts (Mixtral
shape), softmax over all experts with no renormalisation and a sigmoid-gated shared expert
(Qwen1.5-MoE shape), sigmoid scores with a selection-only bias, renormalised and scaled by
2.5, plus an unscaled shared expert (DeepSeek-V3 shape), and the SwiGLU expert FFN
y = (silu(x Wg) * (x Wu)) Wd.

Readings of the unstated details (all are listed with the design notes):
* top-k order: larger score first, ties to the smaller expert id; the chosen set is reported
  in ascending expert id order;
* the intermediate h and the expert outputs y and s are stored as bf16, so the oracle rounds
  them to bf16 (nearest-even) at the same points;
* permutation is stable: within an expert, rows are in ascending token order.
"""
from __future__ import annotations

import numpy as np

from . import bf16

# ----------------------------------------------------------------------------- A1: router


def router_logits(x: np.ndarray, w_r: np.ndarray, logit_bias=None) -> np.ndarray:
    """l[t, e] = sum_h x[t, h] W_r[h, e] (+ b_e), in fp64.  x, w_r as fp64 values."""
    l = np.asarray(x, np.float64) @ np.asarray(w_r, np.float64)
    if logit_bias is not None:
        l = l + np.asarray(logit_bias, np.float64)[None, :]
    return l


def sigmoid(v):
    return 1.0 / (1.0 + np.exp(-np.asarray(v, np.float64)))


# ----------------------------------------------------------------------------- A2: gating


def selection_scores(l: np.ndarray, mode: str, sel_bias=None) -> np.ndarray:
    """The quantity top-k selects on.

    softmax modes: the logits themselves (softmax is monotone).
    sigmoid_bias_renorm: sigmoid(l) + bias (the bias steers selection only).
    """
    if mode in ("softmax_renorm", "softmax"):
        return np.asarray(l, np.float64)
    if mode == "sigmoid_bias_renorm":
        s = sigmoid(l)
        if sel_bias is not None:
            s = s + np.asarray(sel_bias, np.float64)[None, :]
        return s
    raise ValueError(mode)


def topk_select(score: np.ndarray, k: int):
    """Top-k of each row by (score descending, expert id ascending).

    Returns (ids[T, k] int32 in ascending expert id, gap[T]) where gap is the selection
    score of the k-th chosen minus that of the best unchosen expert (inf when k == E).
    """
    T, E = score.shape
    eid = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((eid, -score), axis=-1)      # last key is the primary key
    chosen = np.sort(order[:, :k], axis=1).astype(np.int32)
    if k < E:
        rows = np.arange(T)
        gap = score[rows, order[:, k - 1]] - score[rows, order[:, k]]
    else:
        gap = np.full(T, np.inf)
    return chosen, gap


def gate_weights(l: np.ndarray, ids: np.ndarray, mode: str, scale: float = 1.0) -> np.ndarray:
    """Routed weights w[T, k] for the chosen ids (in the given id order).

    softmax_renorm:      w_j = exp(l_j) / sum_{j' chosen} exp(l_j')
    softmax:             w_j = exp(l_j) / sum_{all e} exp(l_e)
    sigmoid_bias_renorm: w_j = sigmoid(l_j) / sum_{j' chosen} sigmoid(l_j')
    then multiplied by `scale` (2.5 for the DeepSeek-V3 shape, 1 otherwise).
    """
    l = np.asarray(l, np.float64)
    rows = np.arange(l.shape[0])[:, None]
    lc = l[rows, ids]
    if mode == "softmax_renorm":
        m = lc.max(axis=1, keepdims=True)
        e = np.exp(lc - m)
        w = e / e.sum(axis=1, keepdims=True)
    elif mode == "softmax":
        m = l.max(axis=1, keepdims=True)
        w = np.exp(lc - m) / np.exp(l - m).sum(axis=1, keepdims=True)
    elif mode == "sigmoid_bias_renorm":
        s = sigmoid(lc)
        w = s / s.sum(axis=1, keepdims=True)
    else:
        raise ValueError(mode)
    return w * scale


# ----------------------------------------------------------------------------- A3: dispatch


def dispatch(ids: np.ndarray, E: int):
    """Per-expert histogram, exclusive scan and stable destination of every (t, j).

    counts[e]  = #{(t, j) : ids[t, j] == e}
    offsets    = exclusive prefix sum of counts, length E + 1
    pos[t, j]  = offsets[e] + #{(t', j') with ids[t', j'] == e and t' < t}   (e = ids[t, j])
    src[p]     = t * k + j for p = pos[t, j]
    """
    T, k = ids.shape
    counts = np.zeros(E, np.int64)
    for e in ids.reshape(-1):
        counts[int(e)] += 1
    offsets = np.zeros(E + 1, np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    cursor = offsets[:E].copy()
    pos = np.zeros((T, k), np.int64)
    src = np.zeros(T * k, np.int64)
    for t in range(T):               # ascending token order gives the stable order
        for j in range(k):
            e = int(ids[t, j])
            pos[t, j] = cursor[e]
            src[cursor[e]] = t * k + j
            cursor[e] += 1
    return (counts.astype(np.int32), offsets.astype(np.int32), pos.astype(np.int32),
            src.astype(np.int32))


# ----------------------------------------------------------------------------- A4: permute


def permute(x: np.ndarray, src: np.ndarray, k: int) -> np.ndarray:
    """x_perm[p, :] = x[src[p] // k, :]."""
    return np.asarray(x)[np.asarray(src) // k]


# ----------------------------------------------------------------------------- A6-A8: FFN


def dequant_int4(codes: np.ndarray, scales_bits: np.ndarray, group: int) -> np.ndarray:
    """W[r, c] = q[r, c] * scale[r // group, c] along the reduction dimension r, in fp64."""
    q = np.asarray(codes, np.float64)
    s = bf16.decode(scales_bits)
    return q * np.repeat(s, group, axis=0)


# NVFP4.  The expert-cache page names NVFP4 checkpoints ("Running 35B MoE Models on 8GB GPUs",
# "Technical Insight": NVFP4/INT4 scales travel inside the expert bundle) without defining the
# format; the reading here is the published NVFP4 definition: FP4 E2M1 elements, one FP8 E4M3
# scale per 16 consecutive elements, one fp32 scale per tensor.


def decode_e2m1(codes: np.ndarray) -> np.ndarray:
    """FP4 E2M1 nibbles -> fp64: bit 3 sign, bits 2-1 exponent e (bias 1), bit 0 mantissa m;
    value (-1)^sign * (m / 2) for e = 0 (subnormal), else 2^(e - 1) * (1 + m / 2)."""
    c = np.asarray(codes).astype(np.int64)
    sign = np.where((c >> 3) & 1, -1.0, 1.0)
    e = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    mag = np.where(e == 0, m / 2.0, np.ldexp(1.0 + m / 2.0, (e - 1).astype(np.int64)))
    return sign * mag


def decode_e4m3(bytes_: np.ndarray) -> np.ndarray:
    """FP8 E4M3 bytes -> fp64: bit 7 sign, bits 6-3 exponent e (bias 7), bits 2-0 mantissa m;
    (-1)^sign * 2^-6 * (m / 8) for e = 0, else 2^(e - 7) * (1 + m / 8); 0x7F / 0xFF are NaN."""
    b = np.asarray(bytes_).astype(np.int64)
    sign = np.where((b >> 7) & 1, -1.0, 1.0)
    e = (b >> 3) & 15
    m = (b & 7).astype(np.float64)
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64)))
    return np.where((b & 0x7F) == 0x7F, np.nan, sign * mag)


def dequant_nvfp4(codes: np.ndarray, scales: np.ndarray, g: float, block: int = 16) -> np.ndarray:
    """W[r, c] = E2M1(code[r, c]) * E4M3(scale[r // block, c]) * g along the reduction
    dimension r, in fp64 (exact)."""
    return decode_e2m1(codes) * np.repeat(decode_e4m3(scales), block, axis=0) * float(g)


def expert_matrices(w, group: int = 128):
    """(Wg[H, I], Wu[H, I], Wd[I, H]) as fp64 from a workloads.ExpertWeights."""
    if w.wdtype == "bf16":
        return bf16.decode(w.wg), bf16.decode(w.wu), bf16.decode(w.wd)
    if w.wdtype == "nvfp4":
        return (dequant_nvfp4(w.wg, w.sg, w.gs[0]), dequant_nvfp4(w.wu, w.su, w.gs[1]),
                dequant_nvfp4(w.wd, w.sd, w.gs[2]))
    return (dequant_int4(w.wg, w.sg, group), dequant_int4(w.wu, w.su, group),
            dequant_int4(w.wd, w.sd, group))


def swiglu_ffn(xr: np.ndarray, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray):
    """One SwiGLU expert on rows xr[n, H]:  g = xr Wg, u = xr Wu,
    h = bf16(silu(g) * u) with silu(g) = g / (1 + exp(-g)),  y = bf16(h Wd).
    Returns (y, h) as fp64 values of bf16 numbers."""
    xr = np.asarray(xr, np.float64)
    g = xr @ wg
    u = xr @ wu
    h = bf16.round_rne(g / (1.0 + np.exp(-g)) * u)
    y = bf16.round_rne(h @ wd)
    return y, h


# ----------------------------------------------------------------------------- A9: combine


def combine(y_perm: np.ndarray, pos: np.ndarray, w: np.ndarray, shared=None, shared_gate=None):
    """out[t] = bf16( sum_{j=0}^{k-1} w[t, j] y_perm[pos[t, j]] + g_t s[t] ), fp64 inside."""
    T, k = pos.shape
    acc = np.zeros((T, y_perm.shape[1]), np.float64)
    for j in range(k):
        acc += w[:, j:j + 1] * y_perm[pos[:, j]]
    if shared is not None:
        g = np.ones(T) if shared_gate is None else np.asarray(shared_gate, np.float64)
        acc += g[:, None] * shared
    return bf16.round_rne(acc)


# ----------------------------------------------------------------------------- stacked layers


def rms_normalize(x: np.ndarray, eps: float) -> np.ndarray:
    """u[t] = bf16( x[t] / sqrt(mean_h x[t, h]^2 + eps) ), fp64 inside.

    The input of layer l + 1 of a pre-normalised stack of MoE layers (the residual stream
    x_{l+1} = x_l + layer_l(u_l) is RMS-normalised, with no learned scale, before each layer
    after the first).  The pages stream a model layer by layer ("NovaLLM ...", "3. Optimization
    #1 -- Expert-Level Streaming") but do not say how layers are chained; this is the
    pre-normalised residual form of the MoE models the workloads follow."""
    x = np.asarray(x, np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return bf16.round_rne(x / np.sqrt(ms + eps))


# ----------------------------------------------------------------------------- whole layer


def layer_forward(cfg, layer: int, x_bits: np.ndarray, *, forced_ids=None, rows=None,
                  weights=None, shared=None):
    """The whole MoE layer forward for config ``cfg`` (a workloads.MoEConfig).

    x_bits: activations [T, H] bf16 bits.  forced_ids: ids [T, k] to use instead of the
    router's choice (trace injection, or re-running the later steps on another selection).
    rows: optional token indices; routing and dispatch cover all T tokens, the FFN and the
    combine only these tokens (for large shapes).  weights: optional callable
    ``(layer, e, shared) -> ExpertWeights`` (defaults to the seeded generator).

    Returns a dict with logits, scores, ids, gap, w, counts, offsets, pos, src, out (fp64
    values of bf16 numbers, rows of ``rows`` only when given), shared_gate.
    """
    import workloads as wl
    getw = weights or (lambda lay, e, sh=False: wl.expert(cfg, lay, e, shared=sh))
    x = bf16.decode(x_bits)
    T = x.shape[0]
    w_r = wl.router(cfg, layer).astype(np.float64)
    b = wl.popularity_bias(cfg, layer)
    logit_bias = b if cfg.bias_kind == "logit" else None
    sel_bias = b if cfg.bias_kind == "select" else None
    l = router_logits(x, w_r, logit_bias)
    score = selection_scores(l, cfg.gating, sel_bias)
    ids_sel, gap = topk_select(score, cfg.k)
    ids = ids_sel if forced_ids is None else np.asarray(forced_ids, np.int32)
    w = gate_weights(l, ids, cfg.gating, cfg.scale)
    counts, offsets, pos, src = dispatch(ids, cfg.E)

    rows = np.arange(T) if rows is None else np.asarray(rows)
    want = np.zeros(T, bool)
    want[rows] = True
    y_perm = np.zeros((T * cfg.k, cfg.H), np.float64)
    for e in range(cfg.E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        p = np.arange(lo, hi)
        p = p[want[src[p] // cfg.k]]
        if p.size == 0:
            continue
        wg, wu, wd = expert_matrices(getw(layer, e), cfg.group)
        y_perm[p], _ = swiglu_ffn(permute(x, src[p], cfg.k), wg, wu, wd)

    shared_out, g_s = None, None
    if cfg.Is:
        wg, wu, wd = expert_matrices(getw(layer, 0, True), cfg.group)
        shared_out, _ = swiglu_ffn(x[rows], wg, wu, wd)
        if cfg.shared_gate == "sigmoid":
            ws = bf16.decode(wl.shared_gate_vector(cfg, layer))
            g_s = sigmoid(x[rows] @ ws)
    out = combine(y_perm, pos[rows], w[rows], shared_out, g_s)
    return dict(logits=l, scores=score, ids=ids, ids_selected=ids_sel, gap=gap, w=w,
                counts=counts, offsets=offsets, pos=pos, src=src, out=out, rows=rows,
                shared_gate=g_s)


def dense_mixture(x: np.ndarray, gates: np.ndarray, experts) -> np.ndarray:
    """sum_e gates[t, e] * FFN_e(x_t) over every expert (fp64, no bf16 rounding of y).

    Used by the pin that top-k with k == E equals the dense gate-weighted mixture."""
    out = np.zeros_like(np.asarray(x, np.float64))
    for e, (wg, wu, wd) in enumerate(experts):
        g = x @ wg
        u = x @ wu
        out += gates[:, e:e + 1] * ((g / (1.0 + np.exp(-g)) * u) @ wd)
    return out

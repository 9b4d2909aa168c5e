"""Seeded synthetic inputs for the MoE layer forward with expert-slot caching.

This module is shared by the CUDA path's tests and benchmark and by the CPU oracle.  It
only *draws* inputs: tensor shapes, value distributions, routing traces and the per-expert
popularity offsets.  It holds none of the layer's arithmetic (no logits, gating, dispatch,
FFN or combine), so that the oracle and the GPU path share no computation.

Every tensor is drawn from its own NumPy PCG64 stream keyed by
``SeedSequence([seed, cfg_id, a, b, tensor_id, block])``; ``a``/``b`` are (layer, expert)
or (step, layer) depending on the tensor.  Large tensors are split into fixed blocks of
``BLOCK`` elements, each with its own stream, so any one expert can be regenerated alone and
big tensors can be drawn by several threads with identical results.

bf16 values are carried as ``uint16`` bit patterns, rounded from fp32 samples with
round-to-nearest-even.  INT4 weights are carried as ``int8`` codes in [-7, 7] in their
logical layout; NVFP4 weights as ``uint8`` FP4 E2M1 codes (0..15), ``uint8`` FP8 E4M3 block
scales and three fp32 matrix scales; packing into a device bundle is the library's job.

Workload shapes follow the five configurations of the task description (tiny, Mixtral-8x7B
shaped, Qwen1.5-MoE-A2.7B shaped, DeepSeek-V3 shaped INT4, and the expert-streamed decode stack).
"""
from __future__ import annotations

import json
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

BLOCK = 1 << 22

# tensor ids of the stream keys
T_X, T_WR, T_RANK, T_WS, T_TRACE = 0, 1, 2, 3, 4
T_WG, T_WU, T_WD = 10, 11, 12
T_SG, T_SU, T_SD = 20, 21, 22          # INT4 group / NVFP4 block scales of gate / up / down
T_GS = 23                              # NVFP4 matrix scales
T_PROBE = 40                           # calibration batches

GATING = ("softmax_renorm", "softmax", "sigmoid_bias_renorm")


@dataclass(frozen=True)
class MoEConfig:
    """Shape and distribution recipe of one MoE layer workload."""
    name: str
    cfg_id: int
    H: int
    E: int
    k: int
    I: int
    gating: str                 # one of GATING
    scale: float = 1.0          # routed weight multiplier (2.5 for the DeepSeek-V3 shape)
    Is: int = 0                 # shared-expert intermediate size, 0 = none
    shared_gate: str = "none"   # "none" | "sigmoid" (Qwen: sigmoid(x . w_s)) | "one"
    wdtype: str = "bf16"        # "bf16" | "int4_g128" | "nvfp4"
    zipf_s: float = 0.0         # expert-popularity exponent, 0 = no popularity offsets
    bias_kind: str = "none"     # "none" | "logit" (added to logits) | "select" (selection only)
    layers: int = 1
    Ts: tuple = (16,)
    seed: int = 0
    w_std: float = 0.02
    x_std: float = 1.0
    group: int = 128            # INT4 group size along the reduction dimension

    def with_(self, **kw) -> "MoEConfig":
        return replace(self, **kw)


TINY = MoEConfig("tiny", 0, H=256, E=8, k=2, I=512, gating="softmax_renorm", Ts=(16,))
MIXTRAL = MoEConfig("mixtral", 1, H=4096, E=8, k=2, I=14336, gating="softmax_renorm",
                    Ts=(1, 8, 64, 512, 4096))
QWEN = MoEConfig("qwen", 2, H=2048, E=60, k=4, I=1408, gating="softmax", Is=5632,
                 shared_gate="sigmoid", zipf_s=1.0, bias_kind="logit",
                 Ts=(1, 16, 256, 2048, 8192))
DEEPSEEK = MoEConfig("deepseek", 3, H=7168, E=256, k=8, I=2048, gating="sigmoid_bias_renorm",
                     scale=2.5, Is=2048, shared_gate="one", wdtype="int4_g128", zipf_s=1.1,
                     bias_kind="select", Ts=(1, 32, 512, 8192))
# the same Qwen1.5-MoE shape with NVFP4 experts (the checkpoint format the expert-cache page runs)
QWEN_NVFP4 = MoEConfig("qwen_nvfp4", 5, H=2048, E=60, k=4, I=1408, gating="softmax", Is=5632,
                       shared_gate="sigmoid", zipf_s=1.0, bias_kind="logit", wdtype="nvfp4",
                       Ts=(1, 16, 256, 2048, 8192))
STREAMED = MoEConfig("streamed", 4, H=2048, E=60, k=4, I=1408, gating="softmax", Is=5632,
                     shared_gate="sigmoid", zipf_s=1.0, bias_kind="logit", layers=16,
                     Ts=(1, 8, 64))

CONFIGS = {c.name: c for c in (TINY, MIXTRAL, QWEN, DEEPSEEK, STREAMED, QWEN_NVFP4)}

# expert-streamed decode recipe: 256 steps, 4 GiB of VRAM slots, trace locality
STREAM_STEPS = 256
STREAM_CACHE_BYTES = 1 << 32
STREAM_REUSE_P = 0.8
STREAM_TRACE_ZIPF = 1.1
# the stack is pre-normalised: layer l >= 1 takes the residual stream RMS-normalised with this
# epsilon (no learned scale); layer 0 takes the step's unit-scale draw as is
STACK_NORM_EPS = 1e-6

_CAL_PATH = os.path.join(os.path.dirname(__file__), "calibration.json")


def calibration() -> dict:
    """Stored constants written by ``oracle/calibrate_zipf.py`` (only the oracle computes them)."""
    if os.path.exists(_CAL_PATH):
        with open(_CAL_PATH) as f:
            return json.load(f)
    return {}


# ----------------------------------------------------------------------------- streams
def _stream(seed: int, cfg_id: int, a: int, b: int, tensor: int, block: int = 0):
    return np.random.Generator(np.random.PCG64(
        np.random.SeedSequence([seed, cfg_id, a, b, tensor, block])))


_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(32, len(os.sched_getaffinity(0)))))
    return _POOL


def _blocked(n: int, fill, key):
    """Fill an n-element array block by block, each block from its own stream."""
    nb = (n + BLOCK - 1) // BLOCK
    jobs = [(i * BLOCK, min(n, (i + 1) * BLOCK), i) for i in range(nb)]
    if nb == 1:
        return fill(_stream(*key, 0), n)
    parts = list(_pool().map(lambda j: fill(_stream(*key, j[2]), j[1] - j[0]), jobs))
    return np.concatenate(parts)


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round fp32 samples to bf16 (nearest-even), returned as uint16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).reshape(-1)
    out = np.empty(u.size, np.uint16)
    ch = 1 << 20
    for i in range(0, u.size, ch):
        c = u[i:i + ch]
        t = c >> np.uint32(16)
        t &= np.uint32(1)
        t += np.uint32(0x7FFF)
        t += c
        t >>= np.uint32(16)
        out[i:i + ch] = t
    return out.reshape(a.shape)


def _normal_bf16(key, shape, std):
    n = int(np.prod(shape))

    def fill(g, m):
        v = g.standard_normal(m, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        return bf16_bits_from_f32(v)
    return _blocked(n, fill, key).reshape(shape)


def _normal_f32(key, shape, std):
    n = int(np.prod(shape))

    def fill(g, m):
        v = g.standard_normal(m, dtype=np.float32)
        v *= np.float32(std)
        return v
    return _blocked(n, fill, key).reshape(shape)


def _int4_codes(key, shape):
    n = int(np.prod(shape))
    return _blocked(n, lambda g, m: g.integers(-7, 8, m, dtype=np.int8), key).reshape(shape)


def _int4_scales(key, shape, std):
    # symmetric codes uniform in [-7, 7] have variance 56/3; the per-group scale makes the
    # dequantised weight's standard deviation about `std`
    n = int(np.prod(shape))
    base = std / np.sqrt(56.0 / 3.0)

    def fill(g, m):
        v = g.uniform(0.5, 1.5, m).astype(np.float32)
        v *= np.float32(base)
        return bf16_bits_from_f32(v)
    return _blocked(n, fill, key).reshape(shape)


# NVFP4 recipe: E2M1 codes uniform over the 16 nibbles; E4M3 block scales uniform over the
# bytes 0x60..0x7E (32 .. 448: scales near the top of the E4M3 range, as a per-tensor scale
# chosen from the tensor's largest block leaves them); the matrix scale brings the weight's
# standard deviation near `std` (E2M1 uniform: rms 2.93; these scales: rms ~178)
FP4_SCALE_LO, FP4_SCALE_HI = 0x60, 0x7F


def _fp4_codes(key, shape):
    n = int(np.prod(shape))
    return _blocked(n, lambda g, m: g.integers(0, 16, m, dtype=np.uint8), key).reshape(shape)


def _e4m3_scales(key, shape):
    n = int(np.prod(shape))
    return _blocked(n, lambda g, m: g.integers(FP4_SCALE_LO, FP4_SCALE_HI, m, dtype=np.uint8),
                    key).reshape(shape)


def _matrix_scales(key, std):
    g = _stream(*key).uniform(0.75, 1.25, 3)
    return (g * (std / (2.93 * 178.0))).astype(np.float32)


# ----------------------------------------------------------------------------- tensors
def tokens(cfg: MoEConfig, T: int, step: int = 0) -> np.ndarray:
    """Activations x[T, H] as bf16 bits, N(0, x_std)."""
    return _normal_bf16((cfg.seed, cfg.cfg_id, step, T, T_X), (T, cfg.H), cfg.x_std)


def router(cfg: MoEConfig, layer: int = 0) -> np.ndarray:
    """Router weight W_r[H, E] fp32 row-major, N(0, w_std)."""
    return _normal_f32((cfg.seed, cfg.cfg_id, layer, 0, T_WR), (cfg.H, cfg.E), cfg.w_std)


def popularity_ranks(cfg: MoEConfig, layer: int = 0) -> np.ndarray:
    """A per-layer permutation: rank[e] = popularity rank (0 = most popular) of expert e."""
    return _stream(cfg.seed, cfg.cfg_id, layer, 0, T_RANK).permutation(cfg.E).astype(np.int64)


def zipf_probs(E: int, s: float) -> np.ndarray:
    """Zipf(s) probabilities over ranks 0..E-1 (p[r] proportional to (r+1)^-s)."""
    p = np.arange(1, E + 1, dtype=np.float64) ** (-s)
    return p / p.sum()


def popularity_bias(cfg: MoEConfig, layer: int = 0) -> np.ndarray | None:
    """Per-expert offsets b[E] fp32 that give the Zipf(zipf_s) popularity skew.

    ``bias_kind == "logit"``: b_e = ln p_e is added to the router logits (Qwen shape).
    ``bias_kind == "select"``: b_e = beta * ln p_e is added to the sigmoid scores for
    selection only (DeepSeek-V3 shape); beta is the stored calibration constant.
    """
    if cfg.bias_kind == "none" or cfg.zipf_s == 0.0:
        return None
    lp = np.log(zipf_probs(cfg.E, cfg.zipf_s))[popularity_ranks(cfg, layer)]
    if cfg.bias_kind == "select":
        beta = calibration().get(f"beta_{cfg.name}", calibration().get("beta_deepseek", 0.05))
        lp = beta * lp
    return lp.astype(np.float32)


def shared_gate_vector(cfg: MoEConfig, layer: int = 0) -> np.ndarray | None:
    """w_s[H] bf16 bits (Qwen shape: the shared expert is scaled by sigmoid(x . w_s))."""
    if cfg.shared_gate != "sigmoid":
        return None
    return _normal_bf16((cfg.seed, cfg.cfg_id, layer, 0, T_WS), (cfg.H,), cfg.w_std)


@dataclass
class ExpertWeights:
    """Logical weights of one SwiGLU expert.

    bf16: ``wg``/``wu`` [H, I] and ``wd`` [I, H] uint16 bits.
    int4_g128: ``wg``/``wu``/``wd`` int8 codes in the same logical layouts, and bf16 scales
    ``sg``/``su`` [H/group, I] and ``sd`` [I/group, H] (one per group of `group` consecutive
    elements along the reduction dimension).
    nvfp4: ``wg``/``wu``/``wd`` uint8 E2M1 codes, ``sg``/``su`` [H/16, I] and ``sd`` [I/16, H]
    uint8 E4M3 block scales, ``gs`` float32 [3] matrix scales (gate, up, down).
    """
    wdtype: str
    wg: np.ndarray
    wu: np.ndarray
    wd: np.ndarray
    sg: np.ndarray | None = None
    su: np.ndarray | None = None
    sd: np.ndarray | None = None
    gs: np.ndarray | None = None


def expert(cfg: MoEConfig, layer: int, e: int, shared: bool = False) -> ExpertWeights:
    """Weights of routed expert ``e`` of ``layer`` (``shared=True``: the shared expert)."""
    H, I = cfg.H, (cfg.Is if shared else cfg.I)
    eid = cfg.E + 1000 if shared else e
    key = lambda t: (cfg.seed, cfg.cfg_id, layer, eid, t)  # noqa: E731
    if cfg.wdtype == "bf16":
        return ExpertWeights("bf16",
                             _normal_bf16(key(T_WG), (H, I), cfg.w_std),
                             _normal_bf16(key(T_WU), (H, I), cfg.w_std),
                             _normal_bf16(key(T_WD), (I, H), cfg.w_std))
    if cfg.wdtype == "int4_g128":
        G = cfg.group
        assert H % G == 0 and I % G == 0
        return ExpertWeights("int4_g128",
                             _int4_codes(key(T_WG), (H, I)),
                             _int4_codes(key(T_WU), (H, I)),
                             _int4_codes(key(T_WD), (I, H)),
                             _int4_scales(key(T_SG), (H // G, I), cfg.w_std),
                             _int4_scales(key(T_SU), (H // G, I), cfg.w_std),
                             _int4_scales(key(T_SD), (I // G, H), cfg.w_std))
    if cfg.wdtype == "nvfp4":
        assert H % 128 == 0 and I % 128 == 0
        return ExpertWeights("nvfp4",
                             _fp4_codes(key(T_WG), (H, I)),
                             _fp4_codes(key(T_WU), (H, I)),
                             _fp4_codes(key(T_WD), (I, H)),
                             _e4m3_scales(key(T_SG), (H // 16, I)),
                             _e4m3_scales(key(T_SU), (H // 16, I)),
                             _e4m3_scales(key(T_SD), (I // 16, H)),
                             _matrix_scales(key(T_GS), cfg.w_std))
    raise ValueError(cfg.wdtype)


def calibration_tokens(cfg: MoEConfig, T: int) -> np.ndarray:
    """A separate activation batch (seed stream T_PROBE) for offline calibration only."""
    return _normal_bf16((cfg.seed + 1, cfg.cfg_id, 0, T, T_PROBE), (T, cfg.H), cfg.x_std)


# ----------------------------------------------------------------------------- traces
def stream_trace(cfg: MoEConfig, T: int, steps: int = STREAM_STEPS,
                 reuse_p: float = STREAM_REUSE_P, zipf_s: float = STREAM_TRACE_ZIPF) -> np.ndarray:
    """Routing trace of the expert-streamed decode workload: ids[steps, layers, T, k] int32.

    For every (step, layer, token) one Bernoulli(reuse_p) draw decides whether the token
    reuses its previous step's whole expert set at that layer; otherwise k distinct experts
    are drawn one after another without replacement from Zipf(zipf_s) over the layer's
    popularity ranks.  Step 0 always draws.  These ids are an input of the layer call.
    """
    E, k, L = cfg.E, cfg.k, cfg.layers
    ids = np.empty((steps, L, T, k), np.int32)
    p_rank = zipf_probs(E, zipf_s)
    for layer in range(L):
        rank = popularity_ranks(cfg, layer)
        by_rank = np.argsort(rank)              # by_rank[r] = expert with rank r
        g = _stream(cfg.seed, cfg.cfg_id, layer, T, T_TRACE)
        for s in range(steps):
            reuse = g.random(T) < reuse_p
            for t in range(T):
                if s > 0 and reuse[t]:
                    ids[s, layer, t] = ids[s - 1, layer, t]
                    continue
                avail = np.ones(E, bool)
                for j in range(k):
                    pr = p_rank * avail
                    r = int(g.choice(E, p=pr / pr.sum()))
                    avail[r] = False
                    ids[s, layer, t, j] = by_rank[r]
    return ids


def stream_tokens(cfg: MoEConfig, T: int, step: int) -> np.ndarray:
    """Step input of the decode stack x[T, H] bf16 bits, N(0, 1), one stream per step."""
    return _normal_bf16((cfg.seed, cfg.cfg_id, step, T, T_X), (T, cfg.H), 1.0)


def custom(name: str, **kw) -> MoEConfig:
    """A small custom configuration for tests (cfg_id >= 100 keeps its streams separate)."""
    base = dict(cfg_id=100, H=256, E=8, k=2, I=512, gating="softmax_renorm")
    base.update(kw)
    return MoEConfig(name, **base)

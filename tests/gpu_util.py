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

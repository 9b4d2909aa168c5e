"""Writes ``workloads/calibration.json``: the strength of the DeepSeek-V3-shaped selection bias.

Test/bench infrastructure: calls only the oracle and the seeded generators.

The workload asks for Zipf(1.1) expert popularity over 256 experts with top-8 sigmoid
gating.  The selection bias is b_e = beta * ln p_e with p the Zipf(1.1) probabilities over the
layer's popularity ranks.  A per-assignment share of p_1 = 0.207 is not reachable when each
token picks 8 distinct experts (at most 1/8 of the assignments can go to one expert), so the
reading taken here is: beta makes the most popular expert take 1/(2k) = 1/16 of all
assignments (it is chosen by about half of the tokens, 16x the mean load).  beta is found by
bisection on a separate calibration batch (seed + 1, T = 8192) and then frozen.

Usage:  python -m oracle.calibrate_zipf
"""
from __future__ import annotations

import json
import os

import numpy as np

import workloads as wl
from oracle import bf16, moe_ref


def top_share(cfg, l, lp, beta):
    score = moe_ref.selection_scores(l, cfg.gating, beta * lp)
    ids, _ = moe_ref.topk_select(score, cfg.k)
    top = int(np.argmin(wl.popularity_ranks(cfg, 0)))
    return float((ids == top).sum()) / ids.size


def main(T: int = 8192):
    cfg = wl.DEEPSEEK
    x = bf16.decode(wl.calibration_tokens(cfg, T))
    l = moe_ref.router_logits(x, wl.router(cfg, 0))
    lp = np.log(wl.zipf_probs(cfg.E, cfg.zipf_s))[wl.popularity_ranks(cfg, 0)]
    target = 1.0 / (2 * cfg.k)
    lo, hi = 0.0, 1.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if top_share(cfg, l, lp, mid) < target:
            lo = mid
        else:
            hi = mid
    beta = round(0.5 * (lo + hi), 6)
    share = top_share(cfg, l, lp, beta)
    path = os.path.join(os.path.dirname(wl.__file__), "calibration.json")
    data = wl.calibration()
    data.update({"beta_deepseek": beta, "beta_deepseek_top_share": round(share, 6),
                 "beta_deepseek_target_share": target, "calibration_T": T})
    with open(path, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps(data))


if __name__ == "__main__":
    main()

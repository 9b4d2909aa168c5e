"""Host-side checks of the seeded input generators (shapes, determinism, encodings)."""
import numpy as np
import pytest
import torch

import workloads as wl


def test_bf16_encoding_matches_torch():
    v = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 3
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(wl.bf16_bits_from_f32(v), ref)


def test_deterministic_and_blockwise():
    cfg = wl.custom("gen", H=256, I=512)
    a = wl.expert(cfg, 0, 3)
    b = wl.expert(cfg, 0, 3)
    assert np.array_equal(a.wg, b.wg) and np.array_equal(a.wd, b.wd)
    c = wl.expert(cfg, 0, 4)
    assert not np.array_equal(a.wg, c.wg)
    assert a.wg.shape == (256, 512) and a.wd.shape == (512, 256) and a.wg.dtype == np.uint16
    x1 = wl.tokens(cfg, 5)
    assert np.array_equal(x1, wl.tokens(cfg, 5)) and x1.shape == (5, 256)


def test_int4_ranges_and_scale_shapes():
    cfg = wl.custom("gen4", H=256, I=384, wdtype="int4_g128")
    w = wl.expert(cfg, 0, 0)
    assert w.wg.dtype == np.int8 and w.wg.min() >= -7 and w.wg.max() <= 7
    assert w.sg.shape == (2, 384) and w.sd.shape == (3, 256)


def test_router_stats_and_popularity_bias():
    cfg = wl.QWEN
    w = wl.router(cfg, 0)
    assert w.shape == (2048, 60) and w.dtype == np.float32 and abs(w.std() - 0.02) < 1e-3
    b = wl.popularity_bias(cfg, 0)
    r = wl.popularity_ranks(cfg, 0)
    assert np.allclose(b, np.log(wl.zipf_probs(60, 1.0))[r].astype(np.float32))
    assert sorted(r.tolist()) == list(range(60))


def test_stream_trace_locality():
    cfg = wl.STREAMED.with_(layers=2)
    ids = wl.stream_trace(cfg, T=4, steps=50)
    assert ids.shape == (50, 2, 4, 4)
    for s in range(50):
        for l in range(2):
            for t in range(4):
                assert len(set(ids[s, l, t].tolist())) == 4
    reuse = np.mean([np.array_equal(ids[s, l, t], ids[s - 1, l, t])
                     for s in range(1, 50) for l in range(2) for t in range(4)])
    assert 0.7 < reuse < 0.95


def _realised_counts(cfg, T):
    """Expert assignment counts of T tokens routed by the oracle (the workload's own routing)."""
    from oracle import bf16, moe_ref
    x = bf16.decode(wl.tokens(cfg, T))
    b = wl.popularity_bias(cfg, 0)
    l = moe_ref.router_logits(x, wl.router(cfg, 0).astype(np.float64),
                              b if cfg.bias_kind == "logit" else None)
    s = moe_ref.selection_scores(l, cfg.gating, b if cfg.bias_kind == "select" else None)
    ids, _ = moe_ref.topk_select(s, cfg.k)
    return np.bincount(ids.ravel(), minlength=cfg.E), ids.size


def _rank_correlation(a, b):
    """Spearman's rho (no ties handling needed beyond average ranks of equal values)."""
    def ranks(v):
        order = np.argsort(v, kind="stable")
        r = np.empty(len(v))
        r[order] = np.arange(len(v))
        for val in np.unique(v):               # average ranks of ties
            m = v == val
            r[m] = r[m].mean()
        return r
    ra, rb = ranks(np.asarray(a, float)), ranks(np.asarray(b, float))
    return float(np.corrcoef(ra, rb)[0, 1])


@pytest.mark.parametrize("name", ["qwen", "deepseek"])
def test_realised_popularity_follows_the_zipf_ranks(name):
    """The realised expert popularity of a batch routed by the oracle follows the workload's
    Zipf ranks: the most popular rank is the busiest expert, the first ranks' loads decrease,
    popularity and load are strongly rank-correlated, and the busiest expert's share matches
    the workload's definition -- Qwen: Zipf(1.0) over 60 experts as a logit bias, whose top
    probability is 1 / H_60 = 0.214; DeepSeek: the selection bias calibrated (on another batch)
    so that the top expert takes 1 / (2k) = 1/16 of the assignments.  A sign flip, a dropped
    logarithm or a wrong rank permutation in the bias fails one of these."""
    cfg = {"qwen": wl.QWEN, "deepseek": wl.DEEPSEEK}[name]
    cnt, n = _realised_counts(cfg, 2048)
    r = wl.popularity_ranks(cfg, 0)
    by_rank = cnt[np.argsort(r)]
    assert int(np.argmax(cnt)) == int(np.argmin(r))
    assert np.all(np.diff(by_rank[:4]) < 0)
    assert _rank_correlation(-r, cnt) > 0.85
    share = by_rank[0] / n
    if name == "qwen":
        p1 = 1.0 / np.sum(1.0 / np.arange(1, 61))
        assert abs(share - p1) < 0.04, share
    else:
        assert abs(share - 1.0 / 16) < 0.01, share

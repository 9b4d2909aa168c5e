"""Host-side checks of the seeded input generators (shapes, determinism, encodings)."""
import numpy as np
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

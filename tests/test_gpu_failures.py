"""Failure detection of the expert-slot cache, made on the host (no GPU fault, trap or hang).

The cache's copy path has two host-side hooks, read from the environment when a cache is
created: MOE_TEST_DELAY_COPY=n:ms puts a host function that sleeps ms milliseconds on the copy
stream before the n-th miss copy (a slow host link), and MOE_TEST_FAIL_COPY=n makes the n-th
miss copy fail as if it could not be issued.  A bounded host wait must then return
MOE_ERR_TIMEOUT and the cache must work again once the copy stream catches up; a failed copy
must surface as MOE_ERR_CUDA from the layer forward and leave a trace that is still the LRU
policy's (the failed key dropped), with correct outputs once the call is repeated.
"""
import copy

import numpy as np
import pytest
import torch

import workloads as wl
from oracle import bf16, moe_ref
from oracle.lru_sim import LRUSim

from gpu_util import assert_close, oracle_stack, stack_buffers

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import expert_dispatch_streaming_gb300 as m
    return m


@pytest.fixture(scope="module")
def syn(moe):
    from expert_dispatch_streaming_gb300 import synthetic
    return synthetic


def _stack():
    return wl.custom("fstack", cfg_id=132, H=256, E=16, k=4, I=256, gating="softmax", Is=256,
                     shared_gate="sigmoid", zipf_s=1.0, bias_kind="logit", layers=3)


def _cache(moe, syn, cfg, n_slots, timeout_ms, copy_kernel=0):
    store, table = syn.host_bundle_table(cfg, cfg.layers)
    nb = store.shape[1]
    c = moe.moe_expert_cache_config(slot_bytes=nb, capacity_bytes=n_slots * nb,
                                    n_layers=cfg.layers, n_experts=cfg.E, bundles=table,
                                    timeout_ms=timeout_ms, verify_checksums=1, device=0,
                                    copy_kernel=copy_kernel)
    return moe.moe_expert_cache_create(c), store, table


def test_delayed_copy_times_out_then_recovers(moe, syn, monkeypatch):
    cfg = _stack()
    T, steps, n_slots = 3, 3, 40
    monkeypatch.setenv("MOE_TEST_DELAY_COPY", "2:1500")      # the 2nd miss copy waits 1.5 s
    cache, store, table = _cache(moe, syn, cfg, n_slots, timeout_ms=100)
    monkeypatch.delenv("MOE_TEST_DELAY_COPY")
    trace = wl.stream_trace(cfg, T, steps=steps)
    layers = [syn.DeviceLayer(cfg, layer=l, cached=True) for l in range(cfg.layers)]
    ws = layers[0].workspace(T)
    ids = torch.from_numpy(trace).cuda()
    out = None
    bufs = stack_buffers(T, cfg.H)

    def layer(l, s, x, u):
        y, un = bufs[l & 1], bufs[2 + (l & 1)]
        layers[l].forward(u, ws, out=y, forced_ids=ids[s, l], residual=x, cache=cache,
                          out_normed=un)
        return y, un

    try:
        x0 = syn.to_device_bits(wl.stream_tokens(cfg, T, 0))
        x, u = layer(0, 0, x0, x0)
        # the copy stream is held: a bounded wait on it runs out ...
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_expert_cache_sync(cache)
        assert ei.value.status == moe.MOE_ERR_TIMEOUT
        # ... and so does the next layer's routing read-back, queued behind layer 0's misses
        with pytest.raises(moe.MoEError) as ei:
            layer(1, 0, x, u)
        assert ei.value.status == moe.MOE_ERR_TIMEOUT
        torch.cuda.synchronize()                               # the held copy completes
        moe.moe_expert_cache_sync(cache)
        # the timed-out call requested nothing: repeating it continues the stack
        for s in range(steps):
            if s > 0:
                x = u = syn.to_device_bits(wl.stream_tokens(cfg, T, s))
            for l in range(1 if s == 0 else 0, cfg.layers):
                x, u = layer(l, s, x, u)
        torch.cuda.synchronize()
        out = syn.bits_of(x)
        assert moe.moe_workspace_error(ws) == 0
        got = moe.moe_expert_cache_trace(cache)
    finally:
        moe.moe_expert_cache_destroy(cache)
    sim = LRUSim(n_slots)
    for s in range(steps):
        for l in range(cfg.layers):
            sim.request(l, np.unique(trace[s, l]).tolist())
    assert got == sim.trace
    assert_close(out, oracle_stack(cfg, trace, T, steps - 1), "stack after the timeout")


def _sim_request(sim, layer, uniq, state, fail_at):
    """The simulator's side of a request under the fail hook: the request stops at the
    fail_at-th miss (counted over the cache's life), keeps that miss's record and drops its key.
    Returns True when this request failed."""
    probe = copy.deepcopy(sim)
    probe.request(layer, uniq)
    recs = probe.trace[len(sim.trace):]
    for i, r in enumerate(recs):
        if r[3] == 1:
            state["misses"] += 1
            if state["misses"] == fail_at:
                sim.request(layer, uniq[:i + 1])
                sim.evict(layer, uniq[i])
                return True
    sim.request(layer, uniq)
    return False


@pytest.mark.parametrize("copy_kernel", [0, 1])
def test_failed_copy_surfaces_and_keeps_the_trace(moe, syn, monkeypatch, copy_kernel):
    cfg = _stack()
    T, steps, n_slots, fail_at = 3, 4, 9, 7
    monkeypatch.setenv("MOE_TEST_FAIL_COPY", str(fail_at))
    cache, store, table = _cache(moe, syn, cfg, n_slots, timeout_ms=5000,
                                 copy_kernel=copy_kernel)
    monkeypatch.delenv("MOE_TEST_FAIL_COPY")
    trace = wl.stream_trace(cfg, T, steps=steps)
    layers = [syn.DeviceLayer(cfg, layer=l, cached=True) for l in range(cfg.layers)]
    ws = layers[0].workspace(T)
    ids = torch.from_numpy(trace).cuda()
    failed_at = []
    bufs = stack_buffers(T, cfg.H)
    try:
        for s in range(steps):
            x = u = syn.to_device_bits(wl.stream_tokens(cfg, T, s))
            for l in range(cfg.layers):
                y, un = bufs[l & 1], bufs[2 + (l & 1)]
                try:
                    layers[l].forward(u, ws, out=y, forced_ids=ids[s, l], residual=x,
                                      cache=cache, out_normed=un)
                except moe.MoEError as exc:
                    assert exc.status == moe.MOE_ERR_CUDA
                    failed_at.append((s, l))
                    # repeated: the failed key was dropped, so it misses (and copies) again
                    layers[l].forward(u, ws, out=y, forced_ids=ids[s, l], residual=x,
                                      cache=cache, out_normed=un)
                x, u = y, un
        torch.cuda.synchronize()
        out = syn.bits_of(x)
        assert moe.moe_workspace_error(ws) == 0
        got = moe.moe_expert_cache_trace(cache)
        stats = moe.moe_expert_cache_stats(cache)
    finally:
        moe.moe_expert_cache_destroy(cache)
    assert len(failed_at) == 1
    sim = LRUSim(n_slots)
    state = {"misses": 0}
    sim_failed = []
    for s in range(steps):
        for l in range(cfg.layers):
            uniq = np.unique(trace[s, l]).tolist()
            if _sim_request(sim, l, uniq, state, fail_at):
                sim_failed.append((s, l))
                _sim_request(sim, l, uniq, state, fail_at)
    assert sim_failed == failed_at
    assert got == sim.trace
    n_miss = sum(r[3] for r in sim.trace)
    assert stats["misses"] == n_miss
    assert stats["bytes_h2d"] == (n_miss - 1) * store.shape[1]     # the failed copy moved nothing
    assert_close(out, oracle_stack(cfg, trace, T, steps - 1), "stack after the failed copy")

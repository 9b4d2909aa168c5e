"""GPU tests of the expert-slot cache feeding the layer forward.

The cache's hit / miss / eviction / slot trace must equal the LRU simulator's bit for bit, the
stacked layers' outputs must match the oracle, and H2D bytes must equal misses x bundle size.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import bf16, moe_ref
from oracle.lru_sim import LRUSim, CapacityError

from gpu_util import (assert_close, check_stack_layers, oracle_stack, run_stack_step,
                      run_stack_step_recorded, stack_buffers)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import expert_dispatch_streaming_gb300 as m
    return m


@pytest.fixture(scope="module")
def syn(moe):
    from expert_dispatch_streaming_gb300 import synthetic
    return synthetic


def small_stack(layers=4, wdtype="bf16"):
    return wl.custom("stack", cfg_id=130, H=256, E=16, k=4, I=256, gating="softmax", Is=256,
                     shared_gate="sigmoid", zipf_s=1.0, bias_kind="logit", layers=layers,
                     wdtype=wdtype)


def make_cache(moe, syn, cfg, n_slots, timeout_ms=5000, prefetch=0, device_lru=0, copy_kernel=0):
    store, table = syn.host_bundle_table(cfg, cfg.layers)
    nb = store.shape[1]
    c = moe.moe_expert_cache_config(slot_bytes=nb, capacity_bytes=n_slots * nb,
                                    n_layers=cfg.layers, n_experts=cfg.E, bundles=table,
                                    timeout_ms=timeout_ms, verify_checksums=1, device=0,
                                    prefetch_next_layer=prefetch, device_lru=device_lru,
                                    copy_kernel=copy_kernel)
    return moe.moe_expert_cache_create(c), store, table


def run_stack(moe, syn, cfg, cache, trace, T, steps):
    layers = [syn.DeviceLayer(cfg, layer=l, cached=True) for l in range(cfg.layers)]
    ws = layers[0].workspace(T)
    bufs = stack_buffers(T, cfg.H)
    outs = []
    n_missed = 0
    for s in range(steps):
        x = u = syn.to_device_bits(wl.stream_tokens(cfg, T, s))
        for l in range(cfg.layers):
            ids = torch.from_numpy(np.ascontiguousarray(trace[s, l])).cuda()
            y, un = bufs[l & 1], bufs[2 + (l & 1)]
            _, st = layers[l].forward(u, ws, out=y, forced_ids=ids, residual=x, cache=cache,
                                      out_normed=un)
            n_missed += st.n_missed
            x, u = y, un
        torch.cuda.synchronize()
        assert moe.moe_workspace_error(ws) == 0
        outs.append(syn.bits_of(x))
    return outs, n_missed


@pytest.mark.parametrize("mode", ["host", "host_kernel", "prefetch", "prefetch_kernel", "device"])
@pytest.mark.parametrize("T,n_slots", [(1, 6), (3, 12), (5, 40)])
def test_cache_trace_and_outputs_match(moe, syn, T, n_slots, mode):
    """host: the host LRU; prefetch: every layer call also ends with a prefetch request for the
    next layer (predicted from that layer's previous request); *_kernel: misses copied by the
    fill kernel instead of the copy engine; device: the LRU runs on the GPU.  The trace follows
    the simulator and the outputs do not change."""
    cfg = small_stack()
    steps = 6
    prefetch = mode.startswith("prefetch")
    trace = wl.stream_trace(cfg, T, steps=steps)
    cache, store, table = make_cache(moe, syn, cfg, n_slots, prefetch=int(prefetch),
                                     device_lru=int(mode == "device"),
                                     copy_kernel=int(mode.endswith("_kernel")))
    try:
        outs, n_missed = run_stack(moe, syn, cfg, cache, trace, T, steps)
        got = moe.moe_expert_cache_trace(cache)
        stats = moe.moe_expert_cache_stats(cache)
    finally:
        moe.moe_expert_cache_destroy(cache)
    sim = LRUSim(n_slots)
    for s in range(steps):
        for l in range(cfg.layers):
            sim.request(l, np.unique(trace[s, l]).tolist())
            if prefetch:
                sim.prefetch((l + 1) % cfg.layers)
    assert got == sim.trace
    misses = sum(r[3] for r in sim.trace if r[7] == 0)
    fills = sum(r[3] for r in sim.trace if r[7] == 1)
    assert stats["misses"] == misses
    assert n_missed == (misses if mode != "device" else 0)   # the device LRU reports no host count
    assert stats["prefetch_fills"] == fills
    assert (fills > 0) == bool(prefetch)
    assert stats["bytes_h2d"] == (misses + fills) * store.shape[1]
    for s in (0, steps - 1):
        assert_close(outs[s], oracle_stack(cfg, trace, T, s), f"stack step {s}")


def test_cache_capacity_error_and_evict(moe, syn):
    cfg = small_stack(layers=2)
    cache, store, table = make_cache(moe, syn, cfg, 3)
    try:
        used = np.zeros(cfg.E, np.uint8)
        used[[1, 2, 3, 4]] = 1
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_expert_cache_request(cache, 0, used)
        assert ei.value.status == moe.MOE_ERR_CAPACITY
        assert moe.moe_expert_cache_stats(cache)["requests"] == 0
        used[:] = 0
        used[[1, 5, 9]] = 1
        ptrs, nm = moe.moe_expert_cache_request(cache, 0, used)
        assert nm == 3 and sum(p is not None for p in ptrs) == 3
        moe.moe_expert_cache_release(cache, 0)
        moe.moe_expert_cache_evict(cache, 0, 5)
        moe.moe_expert_cache_evict(cache, 0, 7)           # not resident: no-op
        used[:] = 0
        used[[2]] = 1
        ptrs2, nm = moe.moe_expert_cache_request(cache, 0, used)
        assert nm == 1 and ptrs2[2] == ptrs[5]               # the freed slot is reused
        moe.moe_expert_cache_sync(cache)
        # the bundle in the slot is exactly the host bundle (one contiguous copy per miss)
        nb = store.shape[1]
        dev = torch.empty(nb, dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()
        import ctypes
        rt = None
        for name in ("libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so", "libcudart.so"):
            try:
                rt = ctypes.CDLL(name)
                break
            except OSError:
                continue
        assert rt is not None
        rt.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
        assert rt.cudaMemcpy(dev.data_ptr(), ptrs2[2], nb, 3) == 0    # device to device
        torch.cuda.synchronize()
        assert torch.equal(dev.cpu(), store[0 * cfg.E + 2])
    finally:
        moe.moe_expert_cache_destroy(cache)
    sim = LRUSim(3)
    with pytest.raises(CapacityError):
        sim.request(0, [1, 2, 3, 4])


def test_cache_corrupt_bundle_rejected(moe, syn):
    cfg = small_stack(layers=2)
    store, table = syn.host_bundle_table(cfg, cfg.layers)
    store[5, 100] ^= 1
    c = moe.moe_expert_cache_config(slot_bytes=store.shape[1], capacity_bytes=4 * store.shape[1],
                                    n_layers=2, n_experts=cfg.E, bundles=table, timeout_ms=1000,
                                    verify_checksums=1, device=0)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_expert_cache_create(c)
    assert ei.value.status == moe.MOE_ERR_CORRUPT and ei.value.bad_index == 5


def test_explicit_prefetch_and_wait(moe, syn):
    """A caller-driven prefetch: the bundle lands in the slot the simulator predicts, a later
    request hits it (counted as a used prefetch) and waiting for it leaves the bytes intact."""
    cfg = small_stack(layers=2)
    cache, store, table = make_cache(moe, syn, cfg, 4)
    try:
        mask = np.zeros(cfg.E, np.uint8)
        mask[[3, 7]] = 1
        assert moe.moe_expert_cache_prefetch(cache, 1, mask) == 2
        assert moe.moe_expert_cache_prefetch(cache, 0) == 0        # no previous request
        used = np.zeros(cfg.E, np.uint8)
        used[[7, 9]] = 1
        ptrs, nm = moe.moe_expert_cache_request(cache, 1, used)   # waits for the prefetch
        assert nm == 1
        st = moe.moe_expert_cache_stats(cache)
        assert st["prefetch_requests"] == 1 and st["prefetch_fills"] == 2
        assert st["prefetch_used"] == 1 and st["hits"] == 1 and st["misses"] == 1
        moe.moe_expert_cache_sync(cache)
        torch.cuda.synchronize()
        got = moe.moe_expert_cache_trace(cache)
    finally:
        moe.moe_expert_cache_destroy(cache)
    sim = LRUSim(4)
    sim.prefetch(1, [3, 7])
    sim.prefetch(0)
    sim.request(1, [7, 9])
    assert got == sim.trace


def test_device_lru_stack_replays_as_a_cuda_graph(moe, syn):
    """With the LRU on the GPU a whole decode step of the stack (every layer, its cache
    decisions and miss copies) is captured once and replayed: the outputs equal the eager run
    bit for bit and the trace still follows the simulator."""
    cfg = small_stack()
    T, steps, n_slots = 2, 5, 10
    trace = wl.stream_trace(cfg, T, steps=steps)
    cache, store, table = make_cache(moe, syn, cfg, n_slots, device_lru=1)
    layers = [syn.DeviceLayer(cfg, layer=l, cached=True) for l in range(cfg.layers)]
    ws = layers[0].workspace(T)
    x_in = torch.empty((T, cfg.H), dtype=torch.int16, device="cuda")
    ids_in = torch.empty((cfg.layers, T, cfg.k), dtype=torch.int32, device="cuda")
    bufs = stack_buffers(T, cfg.H)
    stream = torch.cuda.Stream()

    def step(c):
        return run_stack_step(layers, ws, x_in, lambda l: ids_in[l], bufs, cache=c,
                              stream=stream)

    outs = []
    try:
        with torch.cuda.stream(stream):
            x_in.copy_(syn.to_device_bits(wl.stream_tokens(cfg, T, 0)))
            ids_in.copy_(torch.from_numpy(np.ascontiguousarray(trace[0])))
            y = step(cache)                  # step 0 eagerly (also warms up the launches)
        stream.synchronize()
        outs.append(syn.bits_of(y).copy())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            y = step(cache)
        for s in range(1, steps):
            with torch.cuda.stream(stream):
                x_in.copy_(syn.to_device_bits(wl.stream_tokens(cfg, T, s)))
                ids_in.copy_(torch.from_numpy(np.ascontiguousarray(trace[s])))
                g.replay()
            stream.synchronize()
            outs.append(syn.bits_of(y).copy())
        assert moe.moe_workspace_error(ws) == 0
        got = moe.moe_expert_cache_trace(cache)
        del g                                # its nodes address this cache's memory
    finally:
        moe.moe_expert_cache_destroy(cache)
    sim = LRUSim(n_slots)
    for s in range(steps):
        for l in range(cfg.layers):
            sim.request(l, np.unique(trace[s, l]).tolist())
    assert got == sim.trace
    # the same steps eagerly, each with a fresh device-LRU cache replaying the same history
    cache2, _, _ = make_cache(moe, syn, cfg, n_slots, device_lru=1)
    try:
        for s in range(steps):
            with torch.cuda.stream(stream):
                x_in.copy_(syn.to_device_bits(wl.stream_tokens(cfg, T, s)))
                ids_in.copy_(torch.from_numpy(np.ascontiguousarray(trace[s])))
                y = step(cache2)
            stream.synchronize()
            assert np.array_equal(syn.bits_of(y), outs[s]), f"step {s}"
    finally:
        moe.moe_expert_cache_destroy(cache2)


def test_device_lru_capacity_error_in_the_error_word(moe, syn):
    cfg = small_stack(layers=1)
    cache, store, table = make_cache(moe, syn, cfg, 2, device_lru=1)
    try:
        layer = syn.DeviceLayer(cfg, layer=0, cached=True)
        T = 4
        ws = layer.workspace(T)
        x = syn.to_device_bits(wl.tokens(cfg, T))
        ids = torch.tensor([[0, 1, 2, 3]] * T, dtype=torch.int32, device="cuda")
        layer.forward(x, ws, forced_ids=ids, cache=cache)
        torch.cuda.synchronize()
        assert moe.moe_workspace_error(ws) == 20
        assert moe.moe_expert_cache_stats(cache)["requests"] == 0
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_expert_cache_request(cache, 0, np.ones(cfg.E, np.uint8))
        assert ei.value.status == moe.MOE_ERR_UNSUPPORTED
    finally:
        moe.moe_expert_cache_destroy(cache)


@pytest.mark.parametrize("mode", ["host_kernel", "device"])
def test_cache_nvfp4_bundles(moe, syn, mode):
    """NVFP4 bundles (codes, block scales and matrix scales in one unit) through the expert
    cache: the trace follows the simulator and the stacked outputs match the oracle."""
    cfg = small_stack(wdtype="nvfp4")
    T, n_slots, steps = 3, 12, 4
    trace = wl.stream_trace(cfg, T, steps=steps)
    cache, store, table = make_cache(moe, syn, cfg, n_slots, device_lru=int(mode == "device"),
                                     copy_kernel=int(mode == "host_kernel"))
    try:
        outs, _ = run_stack(moe, syn, cfg, cache, trace, T, steps)
        got = moe.moe_expert_cache_trace(cache)
    finally:
        moe.moe_expert_cache_destroy(cache)
    sim = LRUSim(n_slots)
    for s_ in range(steps):
        for l in range(cfg.layers):
            sim.request(l, np.unique(trace[s_, l]).tolist())
    assert got == sim.trace
    for s_ in (0, steps - 1):
        assert_close(outs[s_], oracle_stack(cfg, trace, T, s_), f"nvfp4 stack step {s_}")


class _DeviceBytes:
    """A raw device range as a CUDA-array-interface object (torch.as_tensor views it)."""

    def __init__(self, addr, n):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "|u1", "data": (addr, False),
                                         "version": 3}


@pytest.mark.parametrize("copy_kernel", [0, 1])
def test_filled_slots_hold_the_bundles(moe, syn, copy_kernel):
    """The slots a request fills hold the host bundles byte for byte, whether the copy engine
    or the fill kernel copied them."""
    cfg = small_stack(layers=2)
    cache, store, table = make_cache(moe, syn, cfg, 5, copy_kernel=copy_kernel)
    try:
        used = np.zeros(cfg.E, np.uint8)
        used[[0, 3, 7, 15]] = 1
        ptrs, nm = moe.moe_expert_cache_request(cache, 1, used)
        assert nm == 4
        moe.moe_expert_cache_sync(cache)
        nb = store.shape[1]
        for e in (0, 3, 7, 15):
            got = torch.as_tensor(_DeviceBytes(ptrs[e], nb), device="cuda").cpu()
            assert torch.equal(got, store[cfg.E + e].cpu()), f"expert {e}"
    finally:
        moe.moe_expert_cache_destroy(cache)


def test_unreleased_slots_are_not_evicted(moe, syn):
    """Slots a request handed out stay held until the layer is released: a request (or a
    prefetch) that would have to evict one is refused before it changes anything, so a fill
    can never overwrite a bundle whose reads are still enqueued; after the release the same
    request goes through and the trace is the simulator's."""
    cfg = small_stack(layers=2)
    cache, store, table = make_cache(moe, syn, cfg, 2)
    try:
        m01 = np.zeros(cfg.E, np.uint8)
        m01[[1, 2]] = 1
        moe.moe_expert_cache_request(cache, 0, m01)          # slots 0, 1 held by layer 0
        m1 = np.zeros(cfg.E, np.uint8)
        m1[3] = 1
        before = moe.moe_expert_cache_stats(cache)
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_expert_cache_request(cache, 1, m1)       # would evict (0, 1)
        assert ei.value.status == moe.MOE_ERR_CAPACITY
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_expert_cache_prefetch(cache, 1, m1)
        assert ei.value.status == moe.MOE_ERR_CAPACITY
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_expert_cache_evict(cache, 0, 2)
        assert ei.value.status == moe.MOE_ERR_INVALID_ARG
        assert moe.moe_expert_cache_stats(cache) == before
        again = np.zeros(cfg.E, np.uint8)
        again[2] = 1
        moe.moe_expert_cache_request(cache, 0, again)        # a hit evicts nothing: allowed
        moe.moe_expert_cache_release(cache, 0)
        ptrs, nm = moe.moe_expert_cache_request(cache, 1, m1)
        assert nm == 1
        moe.moe_expert_cache_release(cache, 1)
        moe.moe_expert_cache_evict(cache, 0, 2)              # released: allowed
        moe.moe_expert_cache_sync(cache)
        got = moe.moe_expert_cache_trace(cache)
    finally:
        moe.moe_expert_cache_destroy(cache)
    sim = LRUSim(2)
    sim.request(0, [1, 2])
    sim.request(0, [2])
    sim.request(1, [3])
    assert got == sim.trace


# ------------------------------------------------------------------ the expert-streamed stack
# at its stated size: 16 Qwen1.5-MoE-shaped layers, every routed bundle (16.6 GB) in pinned host
# memory, 2^32 bytes of slots (248), 256 decode steps of the seeded locality trace.


@pytest.fixture(scope="module")
def streamed_store(syn):
    cfg = wl.STREAMED
    store, table = syn.host_bundle_table(cfg, cfg.layers)
    layers = [syn.DeviceLayer(cfg, layer=l, cached=True) for l in range(cfg.layers)]
    yield cfg, store, table, layers
    del layers, store


@pytest.mark.parametrize("mode", ["host", "device"])
@pytest.mark.parametrize("T", [1, 8, 64])
def test_streamed_stack_full_size(moe, syn, streamed_store, T, mode):
    """The cache's whole 256-step trace equals the LRU simulator's bit for bit, the copied bytes
    are misses x bundle size, and (T = 1 at steps 0 and 255, T = 8 at step 255) every layer of
    the stack matches the oracle on its own input.  host: the host LRU with misses copied by the
    fill kernel (the benchmark's default path); device: the LRU on the GPU."""
    cfg, store, table, layers = streamed_store
    nb = store.shape[1]
    n_slots = wl.STREAM_CACHE_BYTES // nb
    assert nb == 17301504 and n_slots == 248
    steps = wl.STREAM_STEPS
    trace = wl.stream_trace(cfg, T, steps=steps)
    c = moe.moe_expert_cache_config(slot_bytes=nb, capacity_bytes=wl.STREAM_CACHE_BYTES,
                                    n_layers=cfg.layers, n_experts=cfg.E, bundles=table,
                                    timeout_ms=20000, verify_checksums=0, device=0,
                                    device_lru=int(mode == "device"),
                                    copy_kernel=int(mode == "host"))
    cache = moe.moe_expert_cache_create(c)
    check_steps = {0, steps - 1} if T == 1 else ({steps - 1} if T == 8 else set())
    outs = {}
    try:
        ids_dev = torch.from_numpy(trace).cuda()
        ws = layers[0].workspace(T)
        bufs = stack_buffers(T, cfg.H)
        for s in range(steps):
            x0 = syn.to_device_bits(wl.stream_tokens(cfg, T, s))
            if s in check_steps:
                outs[s] = run_stack_step_recorded(syn, layers, ws, x0, lambda l: ids_dev[s, l],
                                                  bufs, cache=cache)
            else:
                run_stack_step(layers, ws, x0, lambda l: ids_dev[s, l], bufs, cache=cache)
        torch.cuda.synchronize()
        assert moe.moe_workspace_error(ws) == 0
        got = moe.moe_expert_cache_trace(cache)
        stats = moe.moe_expert_cache_stats(cache)
    finally:
        moe.moe_expert_cache_destroy(cache)
    sim = LRUSim(n_slots)
    for s in range(steps):
        for l in range(cfg.layers):
            sim.request(l, np.unique(trace[s, l]).tolist())
    assert len(got) == len(sim.trace)
    assert got == sim.trace
    misses = sum(r[3] for r in sim.trace)
    assert stats["misses"] == misses and stats["hits"] == len(sim.trace) - misses
    assert stats["requests"] == steps * cfg.layers
    assert stats["bytes_h2d"] == misses * nb
    for s, io in sorted(outs.items()):
        check_stack_layers(cfg, trace, s, io, what=f"streamed stack T={T} step {s}")

"""Host-side checks of the C ABI: the library loads, exports every declared entry point, and
its host-only functions (bundle layout / packing, checksum, argument validation, checksum
verification at cache creation) behave as documented.  No GPU is used."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    import expert_dispatch_streaming_gb300 as m
    return m


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(moe):
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(moe._lib, n), n
    assert set(names) == set(moe.EXPORTED)


def test_fnv1a_published_vectors(moe):
    # FNV-1a 64-bit test vectors from the algorithm's published definition
    for s, h in [(b"", 0xcbf29ce484222325), (b"a", 0xaf63dc4c8601ec8c),
                 (b"foobar", 0x85944171f73967e8)]:
        buf = C.create_string_buffer(s, len(s) if s else 1)
        assert moe.moe_checksum64(C.addressof(buf), len(s)) == h


def test_bundle_sizes(moe):
    # C3 shape: 3 * 2048 * 1408 * 2 bytes; C4 shape: INT4 codes + bf16 scales per 128
    assert moe.moe_bundle_bytes(2048, 1408, "bf16") == 17301504
    assert moe.moe_bundle_bytes(7168, 2048, "int4_g128") == 22020096 + 688128
    assert moe.moe_bundle_bytes(4096, 14336, "bf16") == 3 * 4096 * 14336 * 2
    assert moe.moe_bundle_bytes(100, 128, "bf16") == 0


def test_pack_bf16_layout(moe):
    cfg = wl.custom("pk", H=256, I=384)
    w = wl.expert(cfg, 0, 2)
    lay = moe.bundle_layout(256, 384, "bf16")
    buf = np.zeros(lay.total_bytes, np.uint8)
    moe.moe_pack_bundle(256, 384, "bf16", w.wg, w.wu, w.wd, None, None, None, buf)
    gu = buf[lay.gate_up_offset:lay.gate_up_offset + 2 * 384 * 256 * 2].view(np.uint16)
    gu = gu.reshape(2 * 384, 256)
    assert np.array_equal(gu[:384], w.wg.T) and np.array_equal(gu[384:], w.wu.T)
    dn = buf[lay.down_offset:lay.down_offset + 256 * 384 * 2].view(np.uint16).reshape(256, 384)
    assert np.array_equal(dn, w.wd.T)


def test_pack_int4_layout(moe):
    cfg = wl.custom("pk4", H=256, I=384, wdtype="int4_g128")
    w = wl.expert(cfg, 0, 1)
    H, I = 256, 384
    lay = moe.bundle_layout(H, I, "int4_g128")
    buf = np.zeros(lay.total_bytes, np.uint8)
    moe.moe_pack_bundle(H, I, "int4_g128", w.wg, w.wu, w.wd, w.sg, w.su, w.sd, buf)

    def unpack(off, rows, K):
        b = buf[off:off + rows * K // 2].reshape(rows, K // 2)
        lo = (b & 0xF).astype(np.int8)
        hi = (b >> 4).astype(np.int8)
        lo = np.where(lo >= 8, lo - 16, lo)
        hi = np.where(hi >= 8, hi - 16, hi)
        out = np.empty((rows, K), np.int8)
        out[:, 0::2], out[:, 1::2] = lo, hi
        return out
    gu = unpack(lay.gate_up_offset, 2 * I, H)
    assert np.array_equal(gu[:I], w.wg.T) and np.array_equal(gu[I:], w.wu.T)
    assert np.array_equal(unpack(lay.down_offset, H, I), w.wd.T)
    sg = buf[lay.gate_up_scale_offset:lay.gate_up_scale_offset + 2 * I * (H // 128) * 2]
    sg = sg.view(np.uint16).reshape(2 * I, H // 128)
    assert np.array_equal(sg[:I], w.sg.T) and np.array_equal(sg[I:], w.su.T)
    sd = buf[lay.down_scale_offset:lay.down_scale_offset + H * (I // 128) * 2]
    assert np.array_equal(sd.view(np.uint16).reshape(H, I // 128), w.sd.T)


def test_pack_rejects_out_of_range_codes(moe):
    H, I = 128, 128
    q = np.zeros((H, I), np.int8)
    q[3, 4] = -8
    s = np.zeros((1, I), np.uint16)
    buf = np.zeros(moe.moe_bundle_bytes(H, I, "int4_g128"), np.uint8)
    with pytest.raises(moe.MoEError):
        moe.moe_pack_bundle(H, I, "int4_g128", q, q, q, s, s, s, buf)


def test_cache_create_detects_corrupt_bundle_before_any_gpu_work(moe):
    nb, n = 4096, 6
    store = np.random.default_rng(0).integers(0, 256, (n, nb), dtype=np.uint8)
    table = (moe.moe_host_bundle * n)()
    for i in range(n):
        table[i].ptr = store[i].ctypes.data
        table[i].bytes = nb
        table[i].checksum = moe.moe_checksum64(store[i], nb)
    store[4, 1234] ^= 0x10                      # one flipped bit after hashing
    cfg = moe.moe_expert_cache_config(slot_bytes=nb, capacity_bytes=2 * nb, n_layers=2,
                                      n_experts=3, bundles=table, timeout_ms=1000,
                                      verify_checksums=1, device=0)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_expert_cache_create(cfg)
    assert ei.value.status == moe.MOE_ERR_CORRUPT and ei.value.bad_index == 4


def test_argument_validation_without_gpu(moe):
    # k > E, E > 256 and H not a multiple of 8 are rejected before any CUDA call
    for (T, H, E, k) in [(4, 64, 4, 5), (4, 64, 300, 2), (4, 60, 8, 2)]:
        assert moe.moe_route_workspace_size(T, H, E, k) == 0
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_route_topk(1, 1, None, None, None, None, T, H, E, k, 0, 1.0, 1, 1, 1, 1, 1, 1,
                               None, None, None, 1, 1 << 20, 0)
        assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoEError):
        moe.moe_combine(1, 1, 1, 4, 9, 64, None, None, None, 1, 0)

"""Host-side checks of the C ABI: the library loads, exports every declared entry point, and
its host-only functions (bundle layout / packing, checksum, argument validation, checksum
verification at cache creation) behave as documented.  No GPU is used."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import workloads as wl
from oracle import moe_ref

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


def _untile_bf16(buf, rows, K):
    """Inverse of the tiled bf16 image: tiles of 128 rows x 64 k, chunk c of row r at
    r*128 + ((c ^ (r % 8)) * 16) inside the tile."""
    t = buf[:rows * K * 2].view(np.uint16).reshape(rows // 128, K // 64, 128, 8, 8)
    r = np.arange(128)[:, None]
    c = np.arange(8)[None, :]
    src_chunk = c ^ (r % 8)                                  # stored position of chunk c
    out = t[:, :, r, src_chunk, :]                           # [mt, kt, 128, 8, 8]
    return out.transpose(0, 2, 1, 3, 4).reshape(rows, K)


def _untile_int4(buf, rows, K):
    """Inverse of the tiled INT4 image: 8448-byte tiles of 128 rows x 128 k; chunk (c, r) at
    (c*128 + r)*16 holds k = 32c..32c+31 as four 32-bit words; code 8w + 2p + h of word w is
    sign-magnitude, magnitude at bits (4 + 16h + 4p) mod 32 .. +2, sign at bit (15 + 16h + 4p)
    mod 32;
    scales at 8192 + 2r."""
    nt = (rows // 128) * (K // 128)
    t = buf[:nt * 8448].reshape(rows // 128, K // 128, 8448)
    words = t[:, :, :8192].copy().view("<u4").reshape(rows // 128, K // 128, 4, 128, 4)
    words = words.astype(np.int64)                                       # [mt, kt, c, r, word]
    q = np.empty(words.shape + (8,), np.int8)
    for j in range(8):
        p, h = j >> 1, j & 1
        mag = (words >> ((4 + 16 * h + 4 * p) % 32)) & 7
        sgn = (words >> ((15 + 16 * h + 4 * p) % 32)) & 1
        q[..., j] = np.where(sgn == 1, -mag, mag)
    q = q.reshape(words.shape[:4] + (32,))                               # [mt, kt, c, r, 32]
    q = q.transpose(0, 3, 1, 2, 4).reshape(rows, K)
    sc = t[:, :, 8192:8448].copy().view(np.uint16).reshape(rows // 128, K // 128, 128)
    sc = sc.transpose(0, 2, 1).reshape(rows, K // 128)
    return q, sc


def test_pack_bf16_layout(moe):
    H, I = 256, 384
    cfg = wl.custom("pk", H=H, I=I)
    w = wl.expert(cfg, 0, 2)
    lay = moe.bundle_layout(H, I, "bf16")
    buf = np.zeros(lay.total_bytes, np.uint8)
    moe.moe_pack_bundle(H, I, "bf16", w.wg, w.wu, w.wd, None, None, None, buf)
    gu = _untile_bf16(buf[lay.gate_up_offset:], 2 * I, H)
    assert np.array_equal(gu[:I], w.wg.T) and np.array_equal(gu[I:], w.wu.T)
    assert np.array_equal(_untile_bf16(buf[lay.down_offset:], H, I), w.wd.T)
    # hand check of one element: row 130 (tile 1, r = 2), k = 75 (tile 1, chunk 1, elem 3)
    tile = buf[lay.gate_up_offset + (1 * (H // 64) + 1) * 16384:].view(np.uint16)
    assert tile[(2 * 128 + ((1 ^ 2) << 4)) // 2 + 3] == w.wg[75, 130]


def test_pack_int4_layout(moe):
    H, I = 256, 384
    cfg = wl.custom("pk4", H=H, I=I, wdtype="int4_g128")
    w = wl.expert(cfg, 0, 1)
    lay = moe.bundle_layout(H, I, "int4_g128")
    buf = np.zeros(lay.total_bytes, np.uint8)
    moe.moe_pack_bundle(H, I, "int4_g128", w.wg, w.wu, w.wd, w.sg, w.su, w.sd, buf)
    q, sc = _untile_int4(buf[lay.gate_up_offset:], 2 * I, H)
    assert np.array_equal(q[:I], w.wg.T) and np.array_equal(q[I:], w.wu.T)
    assert np.array_equal(sc[:I], w.sg.T) and np.array_equal(sc[I:], w.su.T)
    q, sc = _untile_int4(buf[lay.down_offset:], H, I)
    assert np.array_equal(q, w.wd.T) and np.array_equal(sc, w.sd.T)
    assert lay.total_bytes == 3 * (H // 128) * (I // 128) * 8448


def test_int4_words_decode_as_bf16_subnormals(moe):
    """The documented decode of a code word: rotated right by 4p and masked with 0x80708070,
    pair p of the word is two bf16 subnormals of value q * 2^-129 (low half = the even code)."""
    H, I = 128, 128
    rng = np.random.default_rng(5)
    q = rng.integers(-7, 8, (H, I)).astype(np.int8)
    s = np.full((H // 128, I), 0x3F00, np.uint16)                        # 0.5 is not allowed,
    s[:] = 0x3C00                                                        # 2^-7 is
    buf = np.zeros(moe.moe_bundle_bytes(H, I, "int4_g128"), np.uint8)
    moe.moe_pack_bundle(H, I, "int4_g128", q, q, q, s, s, s, buf)
    words = buf[:8192].view("<u4").astype(np.uint64)                     # tile 0 of gate rows
    for p in range(4):
        rot = ((words >> (4 * p)) | (words << (32 - 4 * p))) & 0xFFFFFFFF if p else words
        v = (rot & 0x80708070).astype(np.uint32)
        lo = ((v & 0xFFFF) << 16).view(np.float32).astype(np.float64) * 2.0 ** 129
        hi = (v & 0xFFFF0000).view(np.float32).astype(np.float64) * 2.0 ** 129
        # word index -> (c, r, w); code k = 32c + 8w + 2p (+1) of row r
        c, r, w = np.unravel_index(np.arange(2048), (4, 128, 4))
        k = 32 * c + 8 * w + 2 * p
        assert np.array_equal(lo, q[k, r].astype(np.float64))
        assert np.array_equal(hi, q[k + 1, r].astype(np.float64))


def _rotr(words, n):
    return ((words >> n) | (words << (32 - n))) & 0xFFFFFFFF if n else words


def _nvfp4_pairs(words):
    """The documented decode of an NVFP4 code word: pairs 0, 1, 2 = the word rotated right by
    0 / 6 / 12 and masked with 0x81C081C0; pair 3 = (rotr 2 & 0x81808180) | (rotr 10 &
    0x00400040).  Returns the four bf16x2 bit patterns (uint32)."""
    w = words.astype(np.uint64)
    out = [(_rotr(w, r) & 0x81C081C0) for r in (0, 6, 12)]
    out.append((_rotr(w, 2) & 0x81808180) | (_rotr(w, 10) & 0x00400040))
    return [o.astype(np.uint32) for o in out]


def _bf16_halves(v):
    lo = ((v & 0xFFFF) << 16).view(np.float32).astype(np.float64)
    hi = (v & 0xFFFF0000).view(np.float32).astype(np.float64)
    return lo, hi


def _untile_nvfp4(buf, rows, K):
    """Inverse of the tiled NVFP4 image through the documented pair decode: 9216-byte tiles of
    128 rows x 128 k; chunk (c, r) at (c*128 + r)*16 holds k = 32c..32c+31 as four words; pair
    p of word w gives codes 8w + 2p (low half) and 8w + 2p + 1 as bf16 numbers of value
    E2M1 * 2^-126; block scales at 8192 + 8r + b.  Returns (values [rows, K], scales
    [rows, K/16])."""
    nt = (rows // 128) * (K // 128)
    t = buf[:nt * 9216].reshape(rows // 128, K // 128, 9216)
    words = t[:, :, :8192].copy().view("<u4").reshape(rows // 128, K // 128, 4, 128, 4)
    vals = np.empty(words.shape + (8,), np.float64)
    for p, v in enumerate(_nvfp4_pairs(words)):
        lo, hi = _bf16_halves(v)
        vals[..., 2 * p] = lo * 2.0 ** 126
        vals[..., 2 * p + 1] = hi * 2.0 ** 126
    vals = vals.reshape(words.shape[:4] + (32,)).transpose(0, 3, 1, 2, 4).reshape(rows, K)
    sc = t[:, :, 8192:9216].reshape(rows // 128, K // 128, 128, 8)
    sc = sc.transpose(0, 2, 1, 3).reshape(rows, K // 16)
    return vals, sc


def test_pack_nvfp4_layout(moe):
    """Every code decodes, by the documented rotations and masks, to E2M1(code) * 2^-126; the
    block scales and matrix scales sit where the layout says."""
    H, I = 256, 384
    cfg = wl.custom("pkf", H=H, I=I, wdtype="nvfp4")
    w = wl.expert(cfg, 0, 3)
    lay = moe.bundle_layout(H, I, "nvfp4")
    buf = np.zeros(lay.total_bytes, np.uint8)
    moe.moe_pack_bundle_nvfp4(H, I, w.wg, w.wu, w.wd, w.sg, w.su, w.sd, w.gs, buf)
    v, sc = _untile_nvfp4(buf[lay.gate_up_offset:], 2 * I, H)
    assert np.array_equal(v[:I], moe_ref.decode_e2m1(w.wg.T))
    assert np.array_equal(v[I:], moe_ref.decode_e2m1(w.wu.T))
    assert np.array_equal(sc[:I], w.sg.T) and np.array_equal(sc[I:], w.su.T)
    v, sc = _untile_nvfp4(buf[lay.down_offset:], H, I)
    assert np.array_equal(v, moe_ref.decode_e2m1(w.wd.T)) and np.array_equal(sc, w.sd.T)
    gs = buf[lay.global_scale_offset:lay.global_scale_offset + 12].view(np.float32)
    assert np.array_equal(gs, w.gs)
    assert lay.gate_up_scale_offset == 8192 and lay.down_scale_offset == lay.down_offset + 8192
    assert lay.down_offset == 2 * (H // 128) * (I // 128) * 9216
    assert lay.total_bytes == lay.global_scale_offset + 256


def test_nvfp4_dequant_product_is_exact(moe):
    """bf16(code placed) * bf16(scale * 2^119) = E2M1 * E4M3 * 2^-7 exactly, for every code and
    every valid scale byte: the product has at most 6 significant bits and stays a normal
    bf16.  (bf16 products emulated in fp64, which is exact for these operands, then checked to
    be representable in bf16.)"""
    codes = np.arange(16)
    scales = np.arange(0x7F)                                            # 0x00 .. 0x7E
    q = moe_ref.decode_e2m1(codes)[:, None]
    s = moe_ref.decode_e4m3(scales)[None, :]
    prod = (q * 2.0 ** -126) * (s * 2.0 ** 119)
    assert np.array_equal(prod, q * s * 2.0 ** -7)
    # representable in bf16: the fp32 rounding of the product keeps only 8 significant bits
    f = prod.astype(np.float32)
    assert np.array_equal(f.astype(np.float64), prod)
    assert np.all((f.view(np.uint32) & 0xFFFF) == 0)
    nz = np.abs(prod[prod != 0])
    assert nz.min() >= 2.0 ** -126 and nz.max() < 2.0 ** 127               # normal range
    # the scale operand as the kernel builds it: the byte shifted left by 4 into a bf16 half
    # reads scale * 2^-120; times 2^120 (exact: back to the scale), times 2^119
    b = scales.astype(np.uint32)
    t = ((b << 4) << 16).view(np.float32).astype(np.float64)            # bf16 half as fp32
    assert np.array_equal(t, moe_ref.decode_e4m3(scales) * 2.0 ** -120)
    B = (t * 2.0 ** 120 * 2.0 ** 119).astype(np.float32)
    assert np.array_equal(B.astype(np.float64), moe_ref.decode_e4m3(scales) * 2.0 ** 119)
    assert np.all(np.isfinite(B)) and np.all((B.view(np.uint32) & 0xFFFF) == 0)


@pytest.mark.parametrize("field,bad", [("code", 16), ("scale", 0x7F), ("scale", 0x80),
                                       ("gs", np.inf), ("gs", 2.0 ** 120), ("gs", np.nan)])
def test_pack_nvfp4_rejects_invalid_inputs(moe, field, bad):
    H, I = 128, 128
    q = np.zeros((H, I), np.uint8)
    s = np.full((H // 16, I), 0x38, np.uint8)
    gs = np.ones(3, np.float32)
    if field == "code":
        q[5, 7] = bad
    elif field == "scale":
        s[3, 9] = bad
    else:
        gs[1] = bad
    buf = np.zeros(moe.moe_bundle_bytes(H, I, "nvfp4"), np.uint8)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_pack_bundle_nvfp4(H, I, q, q, q, s, s, s, gs, buf)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG


def test_generic_packer_refuses_nvfp4(moe):
    H, I = 128, 128
    buf = np.zeros(moe.moe_bundle_bytes(H, I, "nvfp4"), np.uint8)
    q = np.zeros((H, I), np.uint8)
    with pytest.raises(moe.MoEError):
        moe.moe_pack_bundle(H, I, "nvfp4", q, q, q, q, q, q, buf)


@pytest.mark.parametrize("bad", [0x3F00, 0xBF00, 0x7F80, 0x7FC0, 0x4000])
def test_pack_rejects_int4_scales_of_half_or_more(moe, bad):
    """|scale| must stay below 0.5 (and be finite): scale * 2^129 must be a finite bf16."""
    H, I = 128, 128
    q = np.zeros((H, I), np.int8)
    s = np.full((1, I), 0x3C00, np.uint16)
    s[0, 7] = bad
    buf = np.zeros(moe.moe_bundle_bytes(H, I, "int4_g128"), np.uint8)
    with pytest.raises(moe.MoEError):
        moe.moe_pack_bundle(H, I, "int4_g128", q, q, q, s, s, s, buf)
    s[0, 7] = 0x3EFF                                                     # just below 0.5
    moe.moe_pack_bundle(H, I, "int4_g128", q, q, q, s, s, s, buf)


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

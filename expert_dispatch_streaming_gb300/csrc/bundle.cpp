// Expert bundles: layout, host packing and checksum.
//
// A bundle holds everything one SwiGLU expert needs -- its weights and, for INT4 and NVFP4,
// their scales -- as one contiguous block, the unit that is hashed, cached and copied ("Running 35B
// MoE Models on 8GB GPUs: How vvllm-ms Caches Experts in System RAM", section "Technical
// Insight": quantisation metadata travels with the weights as one atomic cache unit).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <stdint.h>
#include <stddef.h>

#include "../../include/moe.h"

namespace {

size_t r256(size_t v) { return (v + 255) / 256 * 256; }

// Tiled bf16 image of the K-major weight rows W[n][k] = src[k][n] (src is K x N row-major):
// tiles of 128 rows x 64 k, tile (mt, kt) at ((mt * K/64) + kt) * 16384 bytes; inside a tile,
// row r's 16-byte chunk c (k = kt*64 + 8c .. +7) sits at r*128 + ((c ^ (r & 7)) << 4), the
// 128-byte-swizzled K-major layout the tensor cores read from shared memory.
void pack_tiled_bf16(const uint16_t* src, size_t K, size_t N, uint16_t* dst) {
  const size_t kt_n = K / 64;
  for (size_t mt = 0; mt < N / 128; ++mt)
    for (size_t kt = 0; kt < kt_n; ++kt) {
      uint16_t* tile = dst + (mt * kt_n + kt) * 8192;
      for (size_t kk = 0; kk < 64; ++kk) {
        const uint16_t* s = src + (kt * 64 + kk) * N + mt * 128;
        const size_t c = kk >> 3, e = kk & 7;
        for (size_t r = 0; r < 128; ++r) tile[r * 64 + (((c ^ (r & 7)) << 3) | e)] = s[r];
      }
    }
}

// Tiled INT4 image of W[n][k] = codes[k][n] with group scales[k/128][n]: tiles of 128 rows x
// 128 k (one scale group), tile (mt, kt) at ((mt * K/128) + kt) * 8448 bytes.  Inside a tile:
// 16-byte chunk (c, r) at (c * 128 + r) * 16 holds codes k = kt*128 + 32c .. +31 of row r as four
// little-endian 32-bit words of eight codes each.  Codes are stored sign-magnitude: in word
// w, code k = 8w + 2p + h (pair p = 0..3, half h = 0/1) keeps its magnitude in bits
// (4 + 16h + 4p) mod 32 .. +2 and its sign in bit (15 + 16h + 4p) mod 32.  Rotating the word
// right by 4p therefore puts pair p's magnitudes at bits 4-6 / 20-22 and signs at bits 15 / 31:
// two bf16 subnormals of value q * 2^-129, which one bf16 multiply by scale * 2^129 turns into
// q * scale.  Then the 128 rows' bf16 scales at 8192 + 2r; |scale| < 0.5 keeps scale * 2^129
// a finite bf16.
bool pack_tiled_int4(const int8_t* codes, const uint16_t* scales, size_t K, size_t N,
                     uint8_t* dst) {
  bool ok = true;
  const size_t kt_n = K / 128;
  for (size_t mt = 0; mt < N / 128; ++mt)
    for (size_t kt = 0; kt < kt_n; ++kt) {
      uint8_t* tile = dst + (mt * kt_n + kt) * 8448;
      for (size_t kk = 0; kk < 128; ++kk) {
        const int8_t* src = codes + (kt * 128 + kk) * N + mt * 128;
        const size_t c = kk >> 5, w = (kk & 31) >> 3, pr = (kk & 7) >> 1, h = kk & 1;
        const unsigned mag_sh = static_cast<unsigned>((4 + 16 * h + 4 * pr) & 31);
        const unsigned sgn_sh = static_cast<unsigned>((15 + 16 * h + 4 * pr) & 31);
        for (size_t r = 0; r < 128; ++r) {
          const int q = src[r];
          ok &= q >= -7 && q <= 7;
          const uint32_t mag = static_cast<uint32_t>(q < 0 ? -q : q) & 7u;
          const uint32_t bits = (mag << mag_sh) | (static_cast<uint32_t>(q < 0) << sgn_sh);
          uint8_t* wp = tile + (c * 128 + r) * 16 + 4 * w;
          uint32_t word;
          std::memcpy(&word, wp, 4);
          word |= bits;
          std::memcpy(wp, &word, 4);
        }
      }
      uint16_t* sc = reinterpret_cast<uint16_t*>(tile + 8192);
      for (size_t r = 0; r < 128; ++r) {
        const uint16_t s = scales[kt * N + mt * 128 + r];
        ok &= ((s >> 7) & 0xFFu) < 126u;   // |scale| < 0.5 and finite
        sc[r] = s;
      }
    }
  return ok;
}

// Bit positions of FP4 code k = 8w + 2p + h inside its 32-bit word, per nibble bit
// (m, e0, e1, sign).  The dequantiser moves pair p to the bf16 positions m 6, e0 7, e1 8,
// sign 15 (+16 for h = 1): pairs 0-2 by one right rotation each (0, 6, 12), pair 3 by two
// (2 for e0, e1 and sign; 10 for m).  The four pairs' bits tile the word.
unsigned fp4_bit(int p, int h, int nib_bit) {
  static const int kTarget[4] = {6, 7, 8, 15};   // m, e0, e1, sign
  static const int kRot[4] = {0, 6, 12, 2};
  const int rot = (p == 3 && nib_bit == 0) ? 10 : kRot[p];
  return static_cast<unsigned>((kTarget[nib_bit] + 16 * h + rot) & 31);
}

// Tiled NVFP4 image of W[n][k] = codes[k][n] with block scales[k/16][n]: tiles of 128 rows x
// 128 k, tile (mt, kt) at ((mt * K/128) + kt) * 9216 bytes; the codes of row r's 32-element
// chunk c at (c * 128 + r) * 16 as four words placed by fp4_bit, then row r's eight E4M3 block
// scales at 8192 + 8r.  Returns false on a code above 15 or a negative / NaN scale.
bool pack_tiled_nvfp4(const uint8_t* codes, const uint8_t* scales, size_t K, size_t N,
                      uint8_t* dst) {
  bool ok = true;
  const size_t kt_n = K / 128;
  for (size_t mt = 0; mt < N / 128; ++mt)
    for (size_t kt = 0; kt < kt_n; ++kt) {
      uint8_t* tile = dst + (mt * kt_n + kt) * 9216;
      for (size_t kk = 0; kk < 128; ++kk) {
        const uint8_t* src = codes + (kt * 128 + kk) * N + mt * 128;
        const size_t c = kk >> 5, w = (kk & 31) >> 3;
        const int pr = static_cast<int>((kk & 7) >> 1), h = static_cast<int>(kk & 1);
        unsigned sh[4];
        for (int b = 0; b < 4; ++b) sh[b] = fp4_bit(pr, h, b);
        for (size_t r = 0; r < 128; ++r) {
          const unsigned q = src[r];
          ok &= q < 16u;
          uint32_t bits = 0;
          for (int b = 0; b < 4; ++b) bits |= static_cast<uint32_t>((q >> b) & 1u) << sh[b];
          uint8_t* wp = tile + (c * 128 + r) * 16 + 4 * w;
          uint32_t word;
          std::memcpy(&word, wp, 4);
          word |= bits;
          std::memcpy(wp, &word, 4);
        }
      }
      for (size_t r = 0; r < 128; ++r)
        for (size_t b = 0; b < 8; ++b) {
          const uint8_t sb = scales[(kt * 8 + b) * N + mt * 128 + r];
          ok &= sb < 0x7Fu;   // sign clear, not NaN
          tile[8192 + 8 * r + b] = sb;
        }
    }
  return ok;
}

}  // namespace

extern "C" {

int moe_bundle_layout_of(int H, int I, int wdtype, moe_bundle_layout* out) {
  if (!out || H <= 0 || I <= 0 || H % 128 || I % 128) return MOE_ERR_INVALID_ARG;
  const size_t h = H, i = I;
  moe_bundle_layout L{};
  if (wdtype == MOE_W_BF16) {
    L.gate_up_offset = 0;
    L.down_offset = r256(2 * i * h * 2);
    L.total_bytes = r256(L.down_offset + h * i * 2);
  } else if (wdtype == MOE_W_INT4_G128) {
    // scales live inside each 8448-byte tile; the scale offsets are those of the first tile
    L.gate_up_offset = 0;
    L.down_offset = r256((2 * i / 128) * (h / 128) * 8448);
    L.gate_up_scale_offset = 8192;
    L.down_scale_offset = L.down_offset + 8192;
    L.total_bytes = r256(L.down_offset + (h / 128) * (i / 128) * 8448);
  } else if (wdtype == MOE_W_NVFP4) {
    L.gate_up_offset = 0;
    L.down_offset = r256((2 * i / 128) * (h / 128) * 9216);
    L.gate_up_scale_offset = 8192;
    L.down_scale_offset = L.down_offset + 8192;
    L.global_scale_offset = r256(L.down_offset + (h / 128) * (i / 128) * 9216);
    L.total_bytes = r256(L.global_scale_offset + 3 * sizeof(float));
  } else {
    return MOE_ERR_INVALID_ARG;
  }
  *out = L;
  return MOE_OK;
}

size_t moe_bundle_bytes(int H, int I, int wdtype) {
  moe_bundle_layout L;
  return moe_bundle_layout_of(H, I, wdtype, &L) == MOE_OK ? L.total_bytes : 0;
}

int moe_pack_bundle(int H, int I, int wdtype, const void* wg, const void* wu, const void* wd,
                    const uint16_t* sg, const uint16_t* su, const uint16_t* sd, void* dst) {
  moe_bundle_layout L;
  if (wdtype == MOE_W_NVFP4 || moe_bundle_layout_of(H, I, wdtype, &L) != MOE_OK || !wg || !wu ||
      !wd || !dst)
    return MOE_ERR_INVALID_ARG;
  char* b = static_cast<char*>(dst);
  std::memset(b, 0, L.total_bytes);
  const size_t h = H, i = I;
  if (wdtype == MOE_W_BF16) {
    uint16_t* gu = reinterpret_cast<uint16_t*>(b + L.gate_up_offset);
    pack_tiled_bf16(static_cast<const uint16_t*>(wg), h, i, gu);          // rows 0..I-1
    pack_tiled_bf16(static_cast<const uint16_t*>(wu), h, i, gu + i * h);  // rows I..2I-1
    pack_tiled_bf16(static_cast<const uint16_t*>(wd), i, h,
                    reinterpret_cast<uint16_t*>(b + L.down_offset));
    return MOE_OK;
  }
  if (!sg || !su || !sd) return MOE_ERR_INVALID_ARG;
  uint8_t* gu = reinterpret_cast<uint8_t*>(b + L.gate_up_offset);
  const size_t half = (i / 128) * (h / 128) * 8448;
  bool ok = pack_tiled_int4(static_cast<const int8_t*>(wg), sg, h, i, gu);
  ok &= pack_tiled_int4(static_cast<const int8_t*>(wu), su, h, i, gu + half);
  ok &= pack_tiled_int4(static_cast<const int8_t*>(wd), sd, i, h,
                        reinterpret_cast<uint8_t*>(b + L.down_offset));
  return ok ? MOE_OK : MOE_ERR_INVALID_ARG;
}

int moe_pack_bundle_nvfp4(int H, int I, const uint8_t* wg, const uint8_t* wu, const uint8_t* wd,
                          const uint8_t* sg, const uint8_t* su, const uint8_t* sd,
                          const float* gs, void* dst) {
  moe_bundle_layout L;
  if (moe_bundle_layout_of(H, I, MOE_W_NVFP4, &L) != MOE_OK || !wg || !wu || !wd || !sg || !su ||
      !sd || !gs || !dst)
    return MOE_ERR_INVALID_ARG;
  for (int j = 0; j < 3; ++j)
    if (!std::isfinite(gs[j]) || std::fabs(gs[j]) >= 0x1p120f) return MOE_ERR_INVALID_ARG;
  uint8_t* b = static_cast<uint8_t*>(dst);
  std::memset(b, 0, L.total_bytes);
  const size_t h = H, i = I;
  const size_t half = (i / 128) * (h / 128) * 9216;
  bool ok = pack_tiled_nvfp4(wg, sg, h, i, b + L.gate_up_offset);
  ok &= pack_tiled_nvfp4(wu, su, h, i, b + L.gate_up_offset + half);
  ok &= pack_tiled_nvfp4(wd, sd, i, h, b + L.down_offset);
  std::memcpy(b + L.global_scale_offset, gs, 3 * sizeof(float));
  return ok ? MOE_OK : MOE_ERR_INVALID_ARG;
}

// FNV-1a, 64-bit (offset basis 14695981039346656037, prime 1099511628211), over bytes.
uint64_t moe_checksum64(const void* data, size_t bytes) {
  const unsigned char* p = static_cast<const unsigned char*>(data);
  uint64_t hsh = 14695981039346656037ull;
  for (size_t n = 0; n < bytes; ++n) {
    hsh ^= p[n];
    hsh *= 1099511628211ull;
  }
  return hsh;
}

}  // extern "C"

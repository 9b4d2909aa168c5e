// Expert bundles: layout, host packing and checksum.
//
// A bundle holds everything one SwiGLU expert needs -- its weights and, for INT4, the group
// scales -- as one contiguous block, the unit that is hashed, cached and copied ("Running 35B
// MoE Models on 8GB GPUs: How vvllm-ms Caches Experts in System RAM", section "Technical
// Insight": quantisation metadata travels with the weights as one atomic cache unit).
#include <algorithm>
#include <cstring>
#include <stdint.h>
#include <stddef.h>

#include "../../include/moe.h"

namespace {

size_t r256(size_t v) { return (v + 255) / 256 * 256; }

// dst[c][r] = src[r][c] for a rows x cols row-major source of 2-byte elements (blocked)
void transpose16(const uint16_t* src, size_t rows, size_t cols, uint16_t* dst) {
  const size_t B = 64;
  for (size_t r0 = 0; r0 < rows; r0 += B)
    for (size_t c0 = 0; c0 < cols; c0 += B) {
      const size_t r1 = std::min(rows, r0 + B), c1 = std::min(cols, c0 + B);
      for (size_t r = r0; r < r1; ++r)
        for (size_t c = c0; c < c1; ++c) dst[c * rows + r] = src[r * cols + c];
    }
}

// INT4 rows of the transposed matrix: dst row c holds src[.][c] for r = 0..rows-1, two codes
// per byte, even r in the low nibble.  Returns false on a code outside [-7, 7].
bool pack_int4_transposed(const int8_t* src, size_t rows, size_t cols, uint8_t* dst) {
  const size_t B = 64;
  bool ok = true;
  for (size_t r0 = 0; r0 < rows; r0 += B)
    for (size_t c0 = 0; c0 < cols; c0 += B) {
      const size_t r1 = std::min(rows, r0 + B), c1 = std::min(cols, c0 + B);
      for (size_t c = c0; c < c1; ++c)
        for (size_t r = r0; r < r1; r += 2) {
          const int8_t lo = src[r * cols + c], hi = src[(r + 1) * cols + c];
          ok &= lo >= -7 && lo <= 7 && hi >= -7 && hi <= 7;
          dst[c * (rows / 2) + r / 2] =
              static_cast<uint8_t>((static_cast<uint8_t>(lo) & 0xFu) |
                                   ((static_cast<uint8_t>(hi) & 0xFu) << 4));
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
    L.gate_up_offset = 0;
    L.down_offset = r256(2 * i * h / 2);
    L.gate_up_scale_offset = r256(L.down_offset + h * i / 2);
    L.down_scale_offset = r256(L.gate_up_scale_offset + 2 * i * (h / 128) * 2);
    L.total_bytes = r256(L.down_scale_offset + h * (i / 128) * 2);
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
  if (moe_bundle_layout_of(H, I, wdtype, &L) != MOE_OK || !wg || !wu || !wd || !dst)
    return MOE_ERR_INVALID_ARG;
  char* b = static_cast<char*>(dst);
  std::memset(b, 0, L.total_bytes);
  const size_t h = H, i = I;
  if (wdtype == MOE_W_BF16) {
    uint16_t* gu = reinterpret_cast<uint16_t*>(b + L.gate_up_offset);
    transpose16(static_cast<const uint16_t*>(wg), h, i, gu);          // rows 0..I-1 = Wg^T
    transpose16(static_cast<const uint16_t*>(wu), h, i, gu + i * h);  // rows I..2I-1 = Wu^T
    transpose16(static_cast<const uint16_t*>(wd), i, h,
                reinterpret_cast<uint16_t*>(b + L.down_offset));      // row h = Wd[:, h]
    return MOE_OK;
  }
  if (!sg || !su || !sd) return MOE_ERR_INVALID_ARG;
  uint8_t* gu = reinterpret_cast<uint8_t*>(b + L.gate_up_offset);
  bool ok = pack_int4_transposed(static_cast<const int8_t*>(wg), h, i, gu);
  ok &= pack_int4_transposed(static_cast<const int8_t*>(wu), h, i, gu + i * (h / 2));
  ok &= pack_int4_transposed(static_cast<const int8_t*>(wd), i, h,
                             reinterpret_cast<uint8_t*>(b + L.down_offset));
  if (!ok) return MOE_ERR_INVALID_ARG;
  // scales, K-major per weight row: row n holds its H/128 (or I/128) group scales
  uint16_t* sgu = reinterpret_cast<uint16_t*>(b + L.gate_up_scale_offset);
  transpose16(sg, h / 128, i, sgu);
  transpose16(su, h / 128, i, sgu + i * (h / 128));
  transpose16(sd, i / 128, h, reinterpret_cast<uint16_t*>(b + L.down_scale_offset));
  return MOE_OK;
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

// Shared device/host helpers of libmoe (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------- status plumbing
void set_cuda_error(cudaError_t e);
int fail_cuda(cudaError_t e);

#define MOE_CUDA_TRY(expr)                                   \
  do {                                                       \
    cudaError_t _e = (expr);                                 \
    if (_e != cudaSuccess) return ::moe::fail_cuda(_e);      \
  } while (0)

#define MOE_LAUNCH_CHECK() MOE_CUDA_TRY(cudaGetLastError())

#define MOE_REQUIRE(cond)                                    \
  do {                                                       \
    if (!(cond)) return MOE_ERR_INVALID_ARG;                 \
  } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// A bump allocator over a caller-provided workspace.
struct WsCursor {
  char* base;
  size_t cap, used;
  explicit WsCursor(void* b, size_t c) : base(static_cast<char*>(b)), cap(c), used(0) {}
  template <class T>
  T* take(size_t n) {
    size_t off = round_up(used, 256);
    used = off + round_up(n * sizeof(T), 256);
    return base ? reinterpret_cast<T*>(base + off) : nullptr;
  }
  bool ok() const { return used <= cap; }
};

int sm_count();

// ---------------------------------------------------------------- programmatic dependent launch
// With MOE_OPT_PDL set, the kernels of the layer are launched with programmatic stream
// serialization (otherwise launch_pdl is a plain launch): a kernel may be
// scheduled while its predecessor in the stream still runs (once every CTA of the predecessor
// has called pdl_trigger), does its own setup, and calls pdl_wait before its first access to
// memory that earlier work writes or reads.  griddepcontrol.wait returns once the predecessor
// grid has completed and its writes are visible; it is a no-op for a kernel launched without a
// programmatic predecessor (after a memset, a copy, or another library's kernel).
extern int g_use_pdl;   // MOE_OPT_PDL
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = g_use_pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
#define MOE_LAUNCH_PDL(kernel, grid, block, smem, st, ...) \
  MOE_CUDA_TRY(::moe::launch_pdl(kernel, grid, block, smem, st, __VA_ARGS__))
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// kernels launched by this thread (the layer forward reports the difference)
extern thread_local long long g_launches;
#define MOE_COUNT_LAUNCH() (++::moe::g_launches)

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
// low half = first element
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ uint32_t float2_to_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // .x = a (low half)
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------- INT4 dequantisation
// The bundle stores INT4 codes sign-magnitude so that pair p of a 32-bit code word, rotated
// right by 4p and masked, is two bf16 subnormals of value q * 2^-129 (magnitude in mantissa
// bits 4-6, sign in bit 15 of each half).  One bf16 multiply by (scale * 2^129) then gives
// bf16(q * scale), rounded once, exactly as a multiply of the integer q by the scale would.
// bf16 arithmetic keeps subnormal operands (there is no flush-to-zero form of it).

// (scale * 2^129) in both halves; exact for every bf16 scale with |scale| < 0.5, which the
// bundle packer enforces.
__device__ __forceinline__ uint32_t int4_scale_pair(uint16_t scale_bits) {
  const float f = bf16_bits_to_float(scale_bits) * 0x1p64f * 0x1p65f;
  const uint32_t b = float_to_bf16_bits(f);
  return b | (b << 16);
}
// Pair p (codes 8w + 2p, 8w + 2p + 1 of code word `word`) -> bf16x2 of q * scale.
template <int P>
__device__ __forceinline__ uint32_t int4_pair(uint32_t word, uint32_t scale_pair) {
  const uint32_t v = (P == 0 ? word : __funnelshift_r(word, word, 4 * P)) & 0x80708070u;
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(v), "r"(scale_pair));
  return d;
}
__device__ __forceinline__ uint32_t int4_pair_dyn(uint32_t word, int p, uint32_t scale_pair) {
  const uint32_t v = __funnelshift_r(word, word, 4 * p) & 0x80708070u;
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(v), "r"(scale_pair));
  return d;
}

// ---------------------------------------------------------------- NVFP4 dequantisation
// The bundle places the bits of each FP4 E2M1 code so that pair p of a 32-bit code word,
// moved by fixed rotations and masks, is two bf16 numbers of value E2M1 * 2^-126 (exponent
// e1 e0 in bf16 exponent bits 8-7, mantissa in bit 6, sign in bit 15: bf16 and E2M1 share
// the same structure up to the exponent bias, 127 against 1).  One bf16 multiply by
// (block scale * 2^119) gives E2M1 * scale * 2^-7, exact: at most 6 significant bits, and a
// normal bf16 for every code and every E4M3 scale.  The matrix scale (times 2^7) is applied
// to the fp32 accumulator.

// (E4M3 scale * 2^119) in both halves of a bf16 pair, for scale byte jb of `four`: a byte
// permute puts the byte in both halves, shifted left by 4 it sits in bf16 exponent / mantissa
// position and reads scale * 2^-120 (E4M3 and bf16 share the structure up to the bias, 7
// against 127, subnormals included); two exact bf16 multiplies by 2^120 and 2^119 give
// scale * 2^119 <= 448 * 2^119 (4 significant bits).  The byte's sign bit is clear (packer).
__device__ __forceinline__ uint32_t fp4_scale_pair(uint32_t four, int jb) {
  const uint32_t t = __byte_perm(four, 0u, jb | 0x40 | (jb << 8) | 0x4000) << 4;
  uint32_t a, d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(t), "r"(0x7B807B80u));   // 2^120
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(0x7B007B00u));   // 2^119
  return d;
}
// Pair p (codes 8w + 2p, 8w + 2p + 1 of code word `word`) -> bf16x2 of E2M1 * scale * 2^-7.
template <int P>
__device__ __forceinline__ uint32_t fp4_pair(uint32_t word, uint32_t scale_pair) {
  uint32_t v;
  if (P == 0) v = word & 0x81C081C0u;
  else if (P == 1) v = __funnelshift_r(word, word, 6) & 0x81C081C0u;
  else if (P == 2) v = __funnelshift_r(word, word, 12) & 0x81C081C0u;
  else v = (__funnelshift_r(word, word, 2) & 0x81808180u) |
           (__funnelshift_r(word, word, 10) & 0x00400040u);
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(v), "r"(scale_pair));
  return d;
}

}  // namespace moe

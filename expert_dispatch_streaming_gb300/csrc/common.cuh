// Shared device/host helpers of libmoe (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

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

}  // namespace moe

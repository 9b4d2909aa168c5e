// Gate-weighted combine / unpermute (A9):
//   out[t] = bf16( sum_{j<k} w[t][j] * y_perm[pos[t][j]] + g_t * s[t] )   (fp32, j in order)
//   optionally out[t] = bf16(residual[t] + out[t]).
// One warp per token row; each lane moves 16-byte vectors (8 bf16) of the k expert rows, the
// shared-expert row and the output, so every access is coalesced and no atomics are used
// (the result does not depend on scheduling).
#include "common.cuh"
#include "route.cuh"

namespace moe {

__global__ void __launch_bounds__(256)
combine_kernel(const uint16_t* __restrict__ y, const int32_t* __restrict__ pos,
               const float* __restrict__ w, int T, int k, int H,
               const uint16_t* __restrict__ shared, const float* __restrict__ shared_gate,
               const uint16_t* __restrict__ residual, uint16_t* __restrict__ out) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (t >= T) return;
  int pj[kMaxK];
  float wj[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    pj[j] = j < k ? pos[(size_t)t * k + j] : 0;
    wj[j] = j < k ? w[(size_t)t * k + j] : 0.f;
  }
  const float gs = shared ? (shared_gate ? shared_gate[t] : 1.f) : 0.f;
  const int nvec = H / 8;
  for (int v = lane; v < nvec; v += 32) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j >= k) break;
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(y + (size_t)pj[j] * H) + v);
      const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = bf16x2_to_float2(qw[i]);
        acc[2 * i] = fmaf(wj[j], f.x, acc[2 * i]);
        acc[2 * i + 1] = fmaf(wj[j], f.y, acc[2 * i + 1]);
      }
    }
    if (shared) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(shared + (size_t)t * H) + v);
      const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = bf16x2_to_float2(qw[i]);
        acc[2 * i] = fmaf(gs, f.x, acc[2 * i]);
        acc[2 * i + 1] = fmaf(gs, f.y, acc[2 * i + 1]);
      }
    }
    uint32_t o[4];
    if (residual) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(residual + (size_t)t * H) + v);
      const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 r = bf16x2_to_float2(qw[i]);
        const float2 b = bf16x2_to_float2(float2_to_bf16x2(acc[2 * i], acc[2 * i + 1]));
        o[i] = float2_to_bf16x2(r.x + b.x, r.y + b.y);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = float2_to_bf16x2(acc[2 * i], acc[2 * i + 1]);
    }
    reinterpret_cast<uint4*>(out + (size_t)t * H)[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

int launch_combine(const uint16_t* y, const int32_t* pos, const float* w, int T, int k, int H,
                   const uint16_t* shared, const float* shared_gate, const uint16_t* residual,
                   uint16_t* out, cudaStream_t st) {
  if (T <= 0) return MOE_OK;
  combine_kernel<<<ceil_div(T * 32, 256), 256, 0, st>>>(y, pos, w, T, k, H, shared,
                                                        shared_gate, residual, out);
  MOE_COUNT_LAUNCH();
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe

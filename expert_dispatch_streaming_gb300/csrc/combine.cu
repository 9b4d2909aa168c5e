// Gate-weighted combine / unpermute (A9):
//   out[t] = bf16( sum_{j<k} w[t][j] * y_perm[pos[t][j]] + g_t * s[t] )   (fp32, j in order)
//   optionally out[t] = bf16(residual[t] + out[t]), and optionally the row RMS-normalised.
// Grid (ceil(H / 1024), min(T, 65535)) of 128-thread blocks: block (c, t) covers elements
// [1024c, 1024c + 1024) of token t (and of t + 65535, ...); each thread moves one 16-byte
// vector (8 bf16) of the k expert rows, the shared-expert row and the output, so every access
// is coalesced and no atomics are used (the result does not depend on scheduling).
#include "common.cuh"
#include "route.cuh"

#include <algorithm>
#include <type_traits>

namespace moe {

constexpr int kCombineThreads = 128;  // one 16-byte vector (8 bf16) per thread

// grid (ceil(H / 1024), T): block (c, t) covers elements [1024c, 1024c + 1024) of token t, so
// every load of a block is issued at once, whatever T is.  K = the top-k, a template
// parameter: the kernel moves a few bytes per instruction, and loops over the eight possible
// expert rows with the unused ones predicated off made it instruction-bound (issue 70% busy at
// 30% of HBM for the Mixtral shape's k = 2).
template <int K>
__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(const uint16_t* __restrict__ y, const int32_t* __restrict__ pos,
               const float* __restrict__ w, int T, int H,
               const uint16_t* __restrict__ shared, const float* __restrict__ shared_gate,
               const uint16_t* __restrict__ residual, uint16_t* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int v = blockIdx.x * kCombineThreads + threadIdx.x;
  if (v >= H / 8) return;
  for (int t = blockIdx.y; t < T; t += gridDim.y) {
  int pj[K];
  float wj[K];
#pragma unroll
  for (int j = 0; j < K; ++j) {
    pj[j] = __ldg(pos + (size_t)t * K + j);
    wj[j] = __ldg(w + (size_t)t * K + j);
  }
  uint4 q[K];
#pragma unroll
  for (int j = 0; j < K; ++j)
    q[j] = __ldg(reinterpret_cast<const uint4*>(y + (size_t)pj[j] * H) + v);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < K; ++j) {
    const uint32_t qw[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = bf16x2_to_float2(qw[i]);
      acc[2 * i] = fmaf(wj[j], f.x, acc[2 * i]);
      acc[2 * i + 1] = fmaf(wj[j], f.y, acc[2 * i + 1]);
    }
  }
  if (shared) {
    const float gs = shared_gate ? __ldg(shared_gate + t) : 1.f;
    const uint4 sq = __ldg(reinterpret_cast<const uint4*>(shared + (size_t)t * H) + v);
    const uint32_t qw[4] = {sq.x, sq.y, sq.z, sq.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = bf16x2_to_float2(qw[i]);
      acc[2 * i] = fmaf(gs, f.x, acc[2 * i]);
      acc[2 * i + 1] = fmaf(gs, f.y, acc[2 * i + 1]);
    }
  }
  uint32_t o[4];
  if (residual) {
    const uint4 rq = __ldg(reinterpret_cast<const uint4*>(residual + (size_t)t * H) + v);
    const uint32_t qw[4] = {rq.x, rq.y, rq.z, rq.w};
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

// The same combine, one block per token row, that also writes the row RMS-normalised:
//   out_n[t] = bf16( out[t] / sqrt(mean_h(out[t][h]^2) + eps) )
// from the bf16 values of out[t] (sum of squares in fp32, block reduction in fixed order), the
// input of the next layer of a pre-norm stack.  Each thread keeps its up to kNormVec vectors of
// the row in registers between the two passes.
constexpr int kNormVec = 4;

__global__ void __launch_bounds__(1024)
combine_norm_kernel(const uint16_t* __restrict__ y, const int32_t* __restrict__ pos,
                    const float* __restrict__ w, int T, int k, int H,
                    const uint16_t* __restrict__ shared, const float* __restrict__ shared_gate,
                    const uint16_t* __restrict__ residual, uint16_t* __restrict__ out,
                    uint16_t* __restrict__ out_n, float eps) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[32];
  const int nv = H / 8;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    int pj[kMaxK];
    float wj[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      pj[j] = j < k ? __ldg(pos + (size_t)t * k + j) : 0;
      wj[j] = j < k ? __ldg(w + (size_t)t * k + j) : 0.f;
    }
    const float gs = (shared && shared_gate) ? __ldg(shared_gate + t) : 1.f;
    uint32_t o[kNormVec][4];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kNormVec; ++i) {
      const int v = threadIdx.x + i * blockDim.x;
      if (v >= nv) break;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int j = 0; j < k; ++j) {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(y + (size_t)pj[j] * H) + v);
        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float2 f = bf16x2_to_float2(qw[c]);
          acc[2 * c] = fmaf(wj[j], f.x, acc[2 * c]);
          acc[2 * c + 1] = fmaf(wj[j], f.y, acc[2 * c + 1]);
        }
      }
      if (shared) {
        const uint4 sq = __ldg(reinterpret_cast<const uint4*>(shared + (size_t)t * H) + v);
        const uint32_t qw[4] = {sq.x, sq.y, sq.z, sq.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float2 f = bf16x2_to_float2(qw[c]);
          acc[2 * c] = fmaf(gs, f.x, acc[2 * c]);
          acc[2 * c + 1] = fmaf(gs, f.y, acc[2 * c + 1]);
        }
      }
      uint4 rq = make_uint4(0, 0, 0, 0);
      if (residual) rq = __ldg(reinterpret_cast<const uint4*>(residual + (size_t)t * H) + v);
      const uint32_t rw[4] = {rq.x, rq.y, rq.z, rq.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t b = float2_to_bf16x2(acc[2 * c], acc[2 * c + 1]);
        if (residual) {
          const float2 r = bf16x2_to_float2(rw[c]);
          const float2 f = bf16x2_to_float2(b);
          b = float2_to_bf16x2(r.x + f.x, r.y + f.y);
        }
        o[i][c] = b;
        const float2 f = bf16x2_to_float2(b);
        ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
      }
      reinterpret_cast<uint4*>(out + (size_t)t * H)[v] = make_uint4(o[i][0], o[i][1], o[i][2],
                                                                    o[i][3]);
    }
    // block sum of squares: warp shuffle tree, then warp 0 over the warps' sums
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
      float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
      if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    const float scale = 1.f / sqrtf(red[0] / (float)H + eps);
    __syncthreads();   // red[0] is rewritten by the next row
#pragma unroll
    for (int i = 0; i < kNormVec; ++i) {
      const int v = threadIdx.x + i * blockDim.x;
      if (v >= nv) break;
      uint32_t n[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float2 f = bf16x2_to_float2(o[i][c]);
        n[c] = float2_to_bf16x2(f.x * scale, f.y * scale);
      }
      reinterpret_cast<uint4*>(out_n + (size_t)t * H)[v] = make_uint4(n[0], n[1], n[2], n[3]);
    }
  }
}

int launch_combine(const uint16_t* y, const int32_t* pos, const float* w, int T, int k, int H,
                   const uint16_t* shared, const float* shared_gate, const uint16_t* residual,
                   uint16_t* out, uint16_t* out_n, float eps, cudaStream_t st) {
  if (T <= 0) return MOE_OK;
  if (out_n) {
    const int nv = H / 8;
    const int threads = std::min(1024, (int)round_up((size_t)ceil_div(nv, kNormVec), 32));
    if (ceil_div(nv, threads) > kNormVec) return MOE_ERR_INVALID_ARG;
    MOE_LAUNCH_PDL(combine_norm_kernel, dim3(std::min(T, 65535)), dim3(threads), 0, st, y, pos,
                   w, T, k, H, shared, shared_gate, residual, out, out_n, eps);
    MOE_COUNT_LAUNCH();
    MOE_LAUNCH_CHECK();
    return MOE_OK;
  }
  dim3 grid(ceil_div(H / 8, kCombineThreads), std::min(T, 65535));
  const dim3 block(kCombineThreads);
  auto go = [&](auto kc) -> int {
    constexpr int K = decltype(kc)::value;
    MOE_LAUNCH_PDL(combine_kernel<K>, grid, block, 0, st, y, pos, w, T, H, shared, shared_gate,
                   residual, out);
    return MOE_OK;
  };
  int r = MOE_ERR_INVALID_ARG;
  switch (k) {
    case 1: r = go(std::integral_constant<int, 1>{}); break;
    case 2: r = go(std::integral_constant<int, 2>{}); break;
    case 3: r = go(std::integral_constant<int, 3>{}); break;
    case 4: r = go(std::integral_constant<int, 4>{}); break;
    case 5: r = go(std::integral_constant<int, 5>{}); break;
    case 6: r = go(std::integral_constant<int, 6>{}); break;
    case 7: r = go(std::integral_constant<int, 7>{}); break;
    case 8: r = go(std::integral_constant<int, 8>{}); break;
    default: break;
  }
  if (r != MOE_OK) return r;
  MOE_COUNT_LAUNCH();
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe

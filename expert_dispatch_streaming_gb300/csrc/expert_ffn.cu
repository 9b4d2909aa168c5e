// Grouped SwiGLU expert FFN, streaming form (A6 gate/up + SiLU*mul, A7 down).
//
// Only the experts a batch selected are touched, each once per batch ("NovaLLM: Running
// Massive MoE Models Fully In-Memory", "3. Optimization #1 -- Expert-Level Streaming"); with
// weights resident the cost becomes memory bandwidth ("Optimization #2 -- Fully In-Memory
// Startup"), so this kernel is organised around streaming every selected weight byte once.
//
// Shape of the computation ("weights as the M operand"): for expert e with n_e rows,
//   D[m][n] = sum_k W_e[m][k] * X[r0 + n][k]
// where m runs over weight rows (intermediate rows for gate/up, hidden rows for down) and n
// over the expert's token rows.  Tokens sit on the narrow N side of mma.m16n8k16, so an expert
// with 1-8 rows wastes nothing on the weight side.
//
// Each thread owns a contiguous 32-element slice of every 128-wide K block: it loads its
// slice of two weight rows with 16-byte loads (a warp covers 8 rows x 64 contiguous bytes per
// load instruction) and the same slice of each token row.  Because the slot -> k assignment
// is the same for A and B, the MMA computes the exact dot product; only the summation order
// changes.  INT4 codes (32 per thread per row = one 16-byte load) are dequantised in registers
// to bf16(code * scale) with the row's group scale (one per 128-block), the same A values the
// tcgen05 kernel builds in shared memory, and multiplied on the tensor cores.
//
// Work unit = (expert with rows, 64-row block of W, K slice).  When there are too few units
// to fill the GPU the K range is split; every split writes fp32 partials and the last CTA to
// finish a (expert, row block) -- found with one atomic counter, no waiting -- sums the splits
// in split order and runs the epilogue, so results do not depend on scheduling.
#include "expert_ffn.cuh"
#include "tc_gemm.cuh"

namespace moe {

int g_ffn_path = 0;

struct GemmKParams {
  const uint16_t* xin;
  const int32_t* offsets;
  const int32_t* active;
  const int32_t* n_active;
  size_t w_off, s_off;
  int K, M, m_blocks, splits, k_per_split, max_rows;
  uint16_t* out;
  float* part;
  int32_t* counters;
  int32_t* err;
  int host_n;
  int16_t host_ids[kMaxExperts];
  BundleTable tab;
  const void* const* dev_tab;
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <bool INT4, bool FUSED, int NT, int U>
__global__ void __launch_bounds__(128) expert_gemm_kernel(const __grid_constant__ GemmKParams p) {
  pdl_trigger();
  pdl_wait();
  constexpr int NR = FUSED ? 4 : 2;   // weight rows per thread: g, g+8 (gate), g, g+8 (up)
  constexpr int VPR = INT4 ? 1 : 4;   // 16-byte vectors per row per 128-block
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tq = lane & 3;
  int u = blockIdx.x;
  const int split = u % p.splits;
  u /= p.splits;
  const int mb = u % p.m_blocks, a = u / p.m_blocks;
  if (a >= (p.host_n >= 0 ? p.host_n : *p.n_active)) return;
  const int e = p.host_n >= 0 ? p.host_ids[a] : p.active[a];
  // the expert's rows, clipped to [0, max_rows) (offsets inconsistent with max_rows are
  // reported as error 8 instead of indexing past the buffers sized by it)
  int r0 = min(max(p.offsets[e], 0), p.max_rows);
  const int ne = max(0, min(p.offsets[e + 1] - p.offsets[e], p.max_rows - r0));
  if (threadIdx.x == 0 && mb == 0 && split == 0 &&
      (r0 != p.offsets[e] || ne != p.offsets[e + 1] - p.offsets[e]))
    atomicExch(p.err, 8);
  const char* bundle = static_cast<const char*>(p.dev_tab ? p.dev_tab[e] : p.tab.p[e]);
  if (ne <= 0 || bundle == nullptr) return;
  const int K = p.K, M = p.M;
  const int m0 = mb * 64 + warp * 16;
  const int k_lo = split * p.k_per_split, k_hi = min(K, k_lo + p.k_per_split);

  // weight row wr lives in row tile wr / 128 at row rr = wr % 128 (tiled bundle layout:
  // bf16 tiles of 128 x 64 k, 128-byte swizzled; INT4 tiles of 128 x 128 k with scales)
  const char* wrow[NR];
  int rsw[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const int wr = m0 + g + 8 * (r & 1) + (r >= 2 ? M : 0);
    const int mt = wr >> 7, rr = wr & 127;
    if (INT4) {
      wrow[r] = bundle + p.w_off + (size_t)mt * (K / 128) * 8448 + rr * 16;
      rsw[r] = rr;
    } else {
      wrow[r] = bundle + p.w_off + (size_t)mt * (K / 64) * 16384 + rr * 128;
      rsw[r] = rr & 7;
    }
  }
  const int MP = FUSED ? 2 * M : M;

  for (int n0 = 0; n0 < ne; n0 += NT * 8) {
    float acc[NT][4], accu[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[j][q] = accu[j][q] = 0.f;

    for (int kb = k_lo; kb < k_hi; kb += 128 * U) {
      uint4 A[U][NR][VPR];
      uint32_t sc[U][NR];   // INT4: (scale * 2^129) pairs of the rows' group scales
#pragma unroll
      for (int uu = 0; uu < U; ++uu) {
        const int kbb = kb + 128 * uu;
        const bool ok = kbb < k_hi;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
#pragma unroll
          for (int v = 0; v < VPR; ++v) {
            const char* ptr =
                INT4 ? wrow[r] + (size_t)(kbb >> 7) * 8448 + tq * 2048
                     : wrow[r] + (size_t)((kbb >> 6) + (tq >> 1)) * 16384 +
                           ((((tq & 1) * 4 + v) ^ rsw[r]) << 4);
            A[uu][r][v] = ok ? ld_stream(ptr) : make_uint4(0, 0, 0, 0);
          }
          sc[uu][r] = (INT4 && ok)
                          ? int4_scale_pair(__ldg(reinterpret_cast<const uint16_t*>(
                                wrow[r] - rsw[r] * 16 + (size_t)(kbb >> 7) * 8448 + 8192) +
                                rsw[r]))
                          : 0u;
        }
      }
#pragma unroll
      for (int uu = 0; uu < U; ++uu) {
        const int kbb = kb + 128 * uu;
        if (kbb >= k_hi) break;
        // A fragments of the 8 k16 steps of this block
        uint32_t af[8][NR][2];
#pragma unroll
        for (int s = 0; s < 8; ++s)
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            if (INT4) {
              // step s uses codes 4s..4s+3 of the thread's 32: word s/2, pairs (s&1)*2, +1
              const uint32_t q = word_of(A[uu][r][0], s >> 1);
              af[s][r][0] = int4_pair_dyn(q, (s & 1) * 2, sc[uu][r]);
              af[s][r][1] = int4_pair_dyn(q, (s & 1) * 2 + 1, sc[uu][r]);
            } else {
              af[s][r][0] = word_of(A[uu][r][s >> 1], (2 * s) & 3);
              af[s][r][1] = word_of(A[uu][r][s >> 1], (2 * s + 1) & 3);
            }
          }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const int n = n0 + 8 * j + g;
          uint4 xb[4];
          const uint4* xp = reinterpret_cast<const uint4*>(
              p.xin + (size_t)(r0 + min(n, ne - 1)) * K + kbb + 32 * tq);
#pragma unroll
          for (int v = 0; v < 4; ++v) xb[v] = n < ne ? __ldg(xp + v) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            const uint32_t b0 = word_of(xb[s >> 1], (2 * s) & 3);
            const uint32_t b1 = word_of(xb[s >> 1], (2 * s + 1) & 3);
            mma_bf16_16816(acc[j], af[s][0][0], af[s][1][0], af[s][0][1], af[s][1][1], b0, b1);
            if (FUSED)
              mma_bf16_16816(accu[j], af[s][2][0], af[s][3][0], af[s][2][1], af[s][3][1], b0,
                             b1);
          }
        }
      }
    }

    // ---- epilogue of this token chunk: D[m][n] with m = m0 + g (+8), n = 8j + 2tq (+1)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int n = n0 + 8 * j + 2 * tq + (q & 1);
        const int m = m0 + g + 8 * (q >> 1);
        if (n >= ne) continue;
        const size_t row = (size_t)(r0 + n);
        if (p.splits == 1) {
          const float v = FUSED ? silu_mul(acc[j][q], accu[j][q]) : acc[j][q];
          p.out[row * M + m] = float_to_bf16_bits(v);
        } else {
          float* pr = p.part + ((size_t)split * p.max_rows + row) * MP;
          pr[m] = acc[j][q];
          if (FUSED) pr[M + m] = accu[j][q];
        }
      }
  }
  if (p.splits == 1) return;

  // ---- split-K: the last CTA of this (expert, row block) sums the splits in order
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t* ctr = p.counters + a * p.m_blocks + mb;
    const int prev = atomicAdd(ctr, 1);
    s_last = prev == p.splits - 1;
    if (s_last) *ctr = 0;  // leave the counter ready for the next launch
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int idx = threadIdx.x; idx < ne * 64; idx += blockDim.x) {
    const int n = idx >> 6, m = mb * 64 + (idx & 63);
    const size_t row = (size_t)(r0 + n);
    float gs = 0.f, us = 0.f;
    for (int sp = 0; sp < p.splits; ++sp) {
      const float* pr = p.part + ((size_t)sp * p.max_rows + row) * MP;
      gs += __ldcg(pr + m);
      if (FUSED) us += __ldcg(pr + M + m);
    }
    p.out[row * M + m] = float_to_bf16_bits(FUSED ? silu_mul(gs, us) : gs);
  }
}

// ------------------------------------------------------------------------------ host side
GemmPlan plan_gemm(const GemmArgs& a) {
  GemmPlan g{};
  g.A_max = std::max(1, std::min(a.E, a.max_rows));
  if (a.host_n >= 0) g.A_max = std::max(1, std::min(g.A_max, a.host_n));
  g.m_blocks = a.M / 64;
  const int avg = ceil_div(std::max(a.max_rows, 1), g.A_max);
  g.nt = avg <= 8 ? 1 : avg <= 16 ? 2 : avg <= 32 ? 4 : 8;
  const int units = g.A_max * g.m_blocks;
  const int target = 4 * sm_count();
  int splits = 1;
  if (units < target) splits = std::min(a.K / 128, ceil_div(target, units));
  g.k_per_split = (int)round_up(ceil_div(a.K, splits), 128);
  g.splits = ceil_div(a.K, g.k_per_split);
  const size_t mp = (size_t)(a.fused ? 2 : 1) * a.M;
  g.part_elems = g.splits > 1 ? (size_t)g.splits * a.max_rows * mp : 0;
  g.counter_elems = g.splits > 1 ? (size_t)g.A_max * g.m_blocks : 0;
  const bool tc_ok = tc_supported(a);
  // INT4 at the smallest batches (at most 64 routed rows, e.g. T <= 8 with k = 8): the
  // streaming kernel's in-register dequantisation beats the tcgen05 kernel's per-step cost;
  // from there on (measured at T = 32 with the DeepSeek-V3 shape) the tcgen05 kernel wins
  const bool int4_decode = a.int4 && a.max_rows <= 64;
  // bf16 with a handful of rows and small expert matrices (measured: the Qwen1.5-MoE shape at
  // T = 1, 4-12 MB per matrix) is launch-cost bound and the streaming kernel is faster there;
  // the Mixtral shape (117-235 MB per matrix) and every larger batch stay on tcgen05
  const double mat_bytes = (double)a.M * a.K * 2.0 * (a.fused ? 2 : 1);
  const bool bf16_tiny = !a.int4 && !a.fp4 && a.max_rows <= 4 && mat_bytes <= 64e6;
  g.use_tc = tc_ok && (g_ffn_path == 2 || (g_ffn_path == 0 && !int4_decode && !bf16_tiny));
  // NVFP4 runs on the tcgen05 kernel only (the streaming kernel has no FP4 decode)
  if (a.fp4) g.use_tc = tc_ok;
  g.tc = plan_tc(a);
  g.part_elems = std::max(g.part_elems, g.tc.part_elems);
  g.counter_elems = std::max(g.counter_elems, g.tc.counter_elems);
  return g;
}

size_t gemm_scratch(WsCursor& c, const GemmPlan& g, float** part, int32_t** counters) {
  float* pp = c.take<float>(std::max<size_t>(g.part_elems, 1));
  int32_t* cc = c.take<int32_t>(std::max<size_t>(g.counter_elems, 1));
  if (part) *part = pp;
  if (counters) *counters = cc;
  return c.used;
}

template <bool INT4, bool FUSED, int U>
static cudaError_t launch_nt(int nt, dim3 grid, const GemmKParams& kp, cudaStream_t st) {
  switch (nt) {
    case 1: return launch_pdl(expert_gemm_kernel<INT4, FUSED, 1, U>, grid, dim3(128), 0, st, kp);
    case 2: return launch_pdl(expert_gemm_kernel<INT4, FUSED, 2, U>, grid, dim3(128), 0, st, kp);
    case 4: return launch_pdl(expert_gemm_kernel<INT4, FUSED, 4, U>, grid, dim3(128), 0, st, kp);
    default: return launch_pdl(expert_gemm_kernel<INT4, FUSED, 8, U>, grid, dim3(128), 0, st, kp);
  }
}

int launch_gemm(const GemmArgs& a, const GemmPlan& g, float* part, int32_t* counters,
                int32_t* err, cudaStream_t st) {
  if (a.max_rows <= 0) return MOE_OK;
  if (g.use_tc) return launch_tc(a, g.tc, part, counters, err, st);
  if (a.fp4) return MOE_ERR_UNSUPPORTED;
  GemmKParams kp{};
  kp.xin = a.xin; kp.offsets = a.offsets; kp.active = a.active; kp.n_active = a.n_active;
  kp.w_off = a.w_off; kp.s_off = a.s_off; kp.K = a.K; kp.M = a.M;
  kp.m_blocks = g.m_blocks; kp.splits = g.splits; kp.k_per_split = g.k_per_split;
  kp.max_rows = a.max_rows; kp.out = a.out; kp.part = part; kp.counters = counters;
  kp.err = err;
  kp.tab = *a.tab;
  kp.dev_tab = a.dev_tab;
  kp.host_n = a.host_n;
  for (int i = 0; i < (a.host_n > 0 ? a.host_n : 0); ++i) kp.host_ids[i] = (int16_t)a.host_ids[i];
  if (a.host_n == 0) return MOE_OK;
  dim3 grid(g.A_max * g.m_blocks * g.splits);
  if (a.int4) {
    if (a.fused) MOE_CUDA_TRY((launch_nt<true, true, 2>(g.nt, grid, kp, st)));
    else MOE_CUDA_TRY((launch_nt<true, false, 4>(g.nt, grid, kp, st)));
  } else {
    if (a.fused) MOE_CUDA_TRY((launch_nt<false, true, 1>(g.nt, grid, kp, st)));
    else MOE_CUDA_TRY((launch_nt<false, false, 2>(g.nt, grid, kp, st)));
  }
  MOE_COUNT_LAUNCH();
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe

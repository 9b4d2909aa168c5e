// Expert FFN kernels' host interface (internal to libmoe).
#pragma once
#include "common.cuh"
#include "route.cuh"

namespace moe {

// Per-expert bundle pointers, passed by value in kernel parameters (2 KB).
struct BundleTable {
  const void* p[kMaxExperts];
};

// One grouped GEMM over the experts that received rows:
//   out[row][m] = epilogue( sum_k W_e[m][k] * xin[row][k] )  for rows of expert e
// FUSED: W_e = gate rows (0..M-1) and up rows (M..2M-1), out = bf16(silu(g) * u) (h, M = I)
// else : W_e = down rows, out = bf16(acc) (y, M = H)
struct GemmArgs {
  const uint16_t* xin;      // [rows][K] bf16
  const int32_t* offsets;   // [E+1]
  const int32_t* active;    // [E]
  const int32_t* n_active;  // [1]
  int host_n;               // >= 0: use host_ids[0..host_n) instead of active/n_active
  const int32_t* host_ids;
  const BundleTable* tab;
  const void* const* dev_tab; // device [E] bundle pointers (device-side cache), else NULL
  size_t w_off, s_off;      // byte offsets of weights/codes and of INT4 scales in a bundle
  long long gs_rel;         // NVFP4: byte offset of the matrix scale(s) from w_off
  int K, M, E;
  int int4, fp4, fused;
  int max_rows;             // upper bound of offsets[E]
  int rows_cap;             // upper bound of one expert's rows (T for a routed batch: a token
                            // picks an expert at most once); 0: max_rows
  uint16_t* out;            // [rows][M]
};

struct TcPlanLite {
  int BN, S, kt_per_split;
  size_t part_elems, counter_elems;
};

struct GemmPlan {
  int A_max;                // upper bound of experts with rows
  int m_blocks, splits, k_per_split, nt;
  size_t part_elems, counter_elems;
  int use_tc;               // 1: tcgen05 kernel, 0: mma.sync streaming kernel
  TcPlanLite tc;
};

// Process-wide choice of the expert FFN kernel: 0 = automatic, 1 = mma.sync streaming kernel,
// 2 = tcgen05 kernel (where supported).
extern int g_ffn_path;

// launch_gemm expects zeroed split-K counters and leaves them zero (see tc_gemm.cuh).
GemmPlan plan_gemm(const GemmArgs& a);
size_t gemm_scratch(WsCursor& c, const GemmPlan& g, float** part, int32_t** counters);
int launch_gemm(const GemmArgs& a, const GemmPlan& g, float* part, int32_t* counters,
                int32_t* err, cudaStream_t st);

}  // namespace moe

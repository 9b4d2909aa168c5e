// tcgen05 grouped expert GEMM: host interface (internal to libmoe).
#pragma once
#include <cuda.h>

#include "expert_ffn.cuh"

namespace moe {

struct TcParams {
  CUtensorMap tmap_b;        // token rows [max_rows][K] bf16, box {64, BN}, 128-byte swizzle
  CUtensorMap tmap_bs;       // quantised weights: the same rows in boxes of {64, 32}, for the
                             // token tiles that are not full
  const int32_t* offsets;
  const int32_t* active;
  const int32_t* n_active;
  int host_n;
  int16_t host_ids[kMaxExperts];
  BundleTable tab;
  const void* const* dev_tab;   // device [E] bundle pointers, read instead of tab when set
  size_t w_off;
  long long gs_rel, gs_rel2;    // NVFP4: matrix scale(s) at section base + gs_rel (group 2: gs_rel2)
  int K, M, S, kt_per_split, max_rows;
  uint16_t* out;
  float* part;
  int32_t* counters;
  int32_t* err;
  // router mode: A is a [M x K] image whose K range repeats the token columns kb_mod k-tiles
  // apart (K = pieces x H); the fp32 result goes to out_f32[row * ldo + m] for m < m_limit
  int kb_mod;
  float* out_f32;
  int ldo, m_limit;
  // optional second group after the routed experts (the shared expert): rows2 token rows of its
  // own token map, with its own weights (section base), shapes, split count and outputs
  int g2;
  CUtensorMap tmap_b2, tmap_bs2;
  const void* w2;
  int M2, K2, S2, kt_per_split2, rows2;
  uint16_t* out2;
  float* part2;
};

using TcPlan = TcPlanLite;

// The launches below expect `counters` (split-K arrival counters) to be zero; every launch
// leaves the counters it used at zero again, so one memset before a sequence of launches
// sharing the array suffices.
bool tc_supported(const GemmArgs& a);
TcPlan plan_tc(const GemmArgs& a);
int launch_tc(const GemmArgs& a, const TcPlan& t, float* part, int32_t* counters, int32_t* err,
              cudaStream_t st);

// One launch for two groups: the routed experts of a1 and one extra group a2 (the shared
// expert: a single expert whose rows are a2.max_rows consecutive token rows).  Both use the
// same kernel variant (token tile, fused or not, weight type); each keeps its own split count.
struct TcPair {
  TcPlan t1, t2;
};
TcPair plan_tc_pair(const GemmArgs& a1, const GemmArgs& a2);
int launch_tc_pair(const GemmArgs& a1, const GemmArgs& a2, const TcPair& pp, float* part1,
                   float* part2, int32_t* counters, int32_t* err, cudaStream_t st);

// Router logits on the tensor cores: logits[t][c] (c < C, fp32, row stride C) =
// sum_k img[c][k] * x[t][k mod H] with img the [Mpad x 3H] tiled bf16 image of the three
// router pieces (see router_prep in route.cu); one group of T rows (offsets {0, T}).  The K
// range is split tc_router_splits(T, H, Mpad) ways; with S > 1 the launch writes only the
// split partials part = [S][T][Mpad] fp32 (split order), which its consumer sums, and leaves
// logits untouched.
int tc_router_splits(int T, int H, int Mpad);
int launch_tc_router(const uint16_t* x, int T, int H, const void* img, int Mpad, int C,
                     const int32_t* meta, float* logits, float* part, int32_t* err,
                     cudaStream_t st);

}  // namespace moe

// tcgen05 grouped expert GEMM: host interface (internal to libmoe).
#pragma once
#include <cuda.h>

#include "expert_ffn.cuh"

namespace moe {

struct TcParams {
  CUtensorMap tmap_b;        // token rows [max_rows][K] bf16, box {64, BN}, 128-byte swizzle
  const int32_t* offsets;
  const int32_t* active;
  const int32_t* n_active;
  int host_n;
  int16_t host_ids[kMaxExperts];
  BundleTable tab;
  size_t w_off;
  int K, M, S, kt_per_split, max_rows;
  uint16_t* out;
  float* part;
  int32_t* counters;
  int32_t* err;
};

using TcPlan = TcPlanLite;

bool tc_supported(const GemmArgs& a);
TcPlan plan_tc(const GemmArgs& a);
int launch_tc(const GemmArgs& a, const TcPlan& t, float* part, int32_t* counters, int32_t* err,
              cudaStream_t st);

}  // namespace moe

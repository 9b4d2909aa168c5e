// Routing kernels' host interface (internal to libmoe).
#pragma once
#include "common.cuh"
#include <algorithm>

namespace moe {

constexpr int kMaxExperts = 256;  // E limit (expert slots per warp lane: 8)
constexpr int kMaxK = 8;          // top-k limit
constexpr int kTileT = 128;       // tokens per dispatch tile (histogram granularity)

struct GateParams {
  const float* part;         // router outputs: S slices [S][T][ldp], C columns used per row
  int S, C, ldp;
  const uint16_t* x;
  const float* w_r;
  const float* w_rT;         // [E][H] transposed router (tensor-core router path) or NULL
  const float* logit_bias;
  const float* sel_bias;
  const int32_t* forced;
  int T, H, E, k, mode;
  float scale;
  int32_t* ids;
  float* w;
  float* logits;
  float* shared_gate;
  int32_t* tie_flags;
  int32_t* hist;
  int tok_per_warp;          // warp-per-token gating: tokens per warp
  int32_t* ids_local;        // or NULL: the chosen ids are also stored here (shared memory)
};

struct RoutePlan {
  int C;            // logit columns (E, + 1 for the shared-expert gate)
  int S;            // H slices of the router product
  int h_per_split;
  int ntiles;       // 128-token dispatch tiles
  int tc;           // 1: router product on the tensor cores (bf16 x 3 pieces), S = 1
  int Mpad;         // rows of the tensor-core router image (C rounded up to 128)
  int tc_S;         // K splits of the tensor-core router product
  int small;        // 1: gating, scan, ranks and row copy in one CTA (T <= kSmallT)
};

// batches of at least this many tokens compute the router product on the tensor cores
constexpr int kTcRouterMinT = 256;
// batches of at most this many tokens run everything after the router product in one CTA
constexpr int kSmallT = 16;
// batches of at least this many tokens gather x_perm in a separate, GPU-wide kernel
constexpr int kSeparateGatherMinT = 1024;
// ... and so do batches whose permuted rows exceed this many bytes (one CTA per 128-token tile
// would copy them)
constexpr size_t kFusedGatherMaxBytes = size_t(512) << 10;

struct RouteScratch {
  float* part;      // [S][T][C]
  int32_t* hist;    // [ntiles][E]
  int32_t* base;    // [ntiles][E]
  int32_t* active;  // [E] experts with rows, ascending
  int32_t* n_active;
  int32_t* shared_meta;  // {0, T, 0, 1}: offsets / active list / count of the shared expert
  uint16_t* img;         // tensor-core router: [Mpad x 3H] tiled bf16 pieces
  float* w_rT;           // tensor-core router: [E][H] fp32
  float* tc_part;        // tensor-core router, tc_S > 1: [tc_S][T][Mpad] fp32 partials
};

struct RouteArgs {
  const uint16_t* x;
  const float* w_r;
  const float* logit_bias;
  const float* sel_bias;
  const uint16_t* w_gate;
  const int32_t* forced;
  int T, H, E, k, gating;
  float scale;
  int32_t *ids, *counts, *offsets, *pos, *src, *tie_flags;
  float *w, *logits, *shared_gate;
  uint16_t* x_perm;  // nullable: fused gather into expert order
  int32_t* err;      // device error word (bounded waits of the tensor-core router)
};

RoutePlan plan_route(int T, int H, int E, int k, bool has_gate);
size_t route_scratch(WsCursor& c, const RoutePlan& r, int T, int E, RouteScratch* out);
int launch_route(const RouteArgs& a, const RoutePlan& r, const RouteScratch& s,
                 cudaStream_t st);
int launch_gather(const uint16_t* x, const int32_t* src, int rows, int k, int H,
                  uint16_t* x_perm, cudaStream_t st);

}  // namespace moe

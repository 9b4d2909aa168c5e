// Fused small-batch (decode) layer forward: host interface (internal to libmoe).
#pragma once
#include "common.cuh"
#include "expert_ffn.cuh"
#include "route.cuh"

namespace moe {

// batches of at most this many tokens (and every bundle resident) run the whole layer in one
// cooperative launch
constexpr int kDecodeMaxT = kSmallT;

struct DecodePlan {
  int ok;                  // 1: the shape is supported
  int grid;                // CTAs (all resident: cooperative launch)
  int S, hps;              // router H slices and rows per slice
  int C, Cp;               // router columns (E, + 1 for the shared-expert gate); C rounded
                           // up to 4 (the row pitch of the router partials)
  int Umax;                // upper bound of experts with rows, min(E, T*k)
  int Sg, Sd, Sgs, Sds;    // K splits: routed gate/up, routed down, shared gate/up, shared down
  int NB;                  // 256-column blocks of H (combine / normalisation units)
  size_t gpart_elems, dpart_elems, ctl_words;
};

struct DecodeArgs {
  const uint16_t* x;         // [T][H] layer input
  const uint16_t* residual;  // [T][H] or NULL
  const int32_t* forced;     // [T][k] or NULL
  const float *w_r, *logit_bias, *sel_bias;
  const uint16_t* w_gate;    // shared-expert gate vector or NULL
  int T, H, E, k, I, Is, gating, wdtype, shared_sigmoid;
  float scale, eps;
  BundleTable tab;           // routed bundles
  const void* shared;        // shared bundle or NULL
  moe_bundle_layout lay, slay;
  // outputs
  uint16_t* out;
  uint16_t* out_n;           // or NULL
  int32_t *ids, *counts, *offsets, *pos, *src, *tie, *active, *n_active;
  float *w, *shared_gate;
  // scratch
  float *part, *gpart, *dpart, *ss;
  uint16_t *h, *y, *hs, *ys;
  int32_t* ctl;              // ctl_words, zero on entry
  int32_t* err;
};

DecodePlan plan_decode(int T, int H, int E, int k, int I, int Is, int wdtype, bool has_gate);
int launch_decode(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st);

}  // namespace moe

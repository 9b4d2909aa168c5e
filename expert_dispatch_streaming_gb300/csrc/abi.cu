// C-ABI entry points of libmoe and the whole-layer forward.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <functional>
#include <vector>

#include "cache.h"
#include "common.cuh"
#include "decode.cuh"
#include "expert_ffn.cuh"
#include "route.cuh"
#include "tc_gemm.cuh"

namespace moe {

static thread_local int g_last_cuda = 0;
int g_decode_path = 1;   // MOE_OPT_DECODE_KERNEL: 0 off, 1 auto, 2 always
int g_use_pdl = 0;
thread_local long long g_launches = 0;

void set_cuda_error(cudaError_t e) { g_last_cuda = (int)e; }
int fail_cuda(cudaError_t e) {
  set_cuda_error(e);
  return MOE_ERR_CUDA;
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  }
  return n;
}

int launch_combine(const uint16_t* y, const int32_t* pos, const float* w, int T, int k, int H,
                   const uint16_t* shared, const float* shared_gate, const uint16_t* residual,
                   uint16_t* out, uint16_t* out_n, float eps, cudaStream_t st);

// largest row length the fused RMS normalisation of the combine takes (1024 threads x 4
// vectors of 8 elements)
constexpr int kMaxNormH = 32768;

static bool valid_route_shape(int T, int H, int E, int k) {
  return T >= 0 && H > 0 && H % 8 == 0 && E > 0 && E <= kMaxExperts && k >= 1 &&
         k <= std::min(E, kMaxK);
}

// ------------------------------------------------------------------ layer plan
struct LayerScratch {
  RouteScratch rs;
  int32_t *ids, *counts, *offsets, *pos, *src, *tie;
  float *w, *shared_gate;
  uint16_t *x_perm, *h, *y_perm, *h_s, *s;
  float* part;
  float* part_s;    // split-K partials of the shared expert when it shares a launch
  float *dec_rpart, *dec_gpart, *dec_dpart, *dec_ss;   // fused decode kernel scratch
  int32_t* counters;
  int32_t* err;     // device error word (first bytes of the workspace)
  size_t ctl_bytes; // bytes of the control block at the start of the workspace
};

struct LayerPlan {
  RoutePlan rp;
  GemmPlan gu, dn, sgu, sdn;
  moe_bundle_layout lay, slay;
  int merged;        // routed and shared expert share one tcgen05 launch per GEMM
  TcPair mgu, mdn;
  DecodePlan dec;    // the fused decode kernel (small batches, resident bundles)
};

static GemmArgs gemm_args(const moe_bundle_layout& lay, int wdtype, bool fused, int K, int M,
                          int E, int max_rows, int rows_cap = 0) {
  GemmArgs a{};
  a.rows_cap = rows_cap;
  a.K = K;
  a.M = M;
  a.E = E;
  a.int4 = wdtype == MOE_W_INT4_G128;
  a.fp4 = wdtype == MOE_W_NVFP4;
  a.fused = fused;
  a.max_rows = max_rows;
  a.w_off = fused ? lay.gate_up_offset : lay.down_offset;
  a.s_off = fused ? lay.gate_up_scale_offset : lay.down_scale_offset;
  // NVFP4 matrix scales: gate, up, down fp32 at global_scale_offset
  a.gs_rel = a.fp4 ? (long long)lay.global_scale_offset + (fused ? 0 : 8) - (long long)a.w_off : 0;
  a.host_n = -1;
  return a;
}

static int make_plan(const moe_layer* L, int T, LayerPlan* P) {
  if (!L || !valid_route_shape(T, L->H, L->E, L->k) || L->I <= 0 || L->I % 128 ||
      L->H % 128 || L->Is < 0 || L->Is % 128)
    return MOE_ERR_INVALID_ARG;
  if (moe_bundle_layout_of(L->H, L->I, L->wdtype, &P->lay) != MOE_OK) return MOE_ERR_INVALID_ARG;
  if (L->Is && moe_bundle_layout_of(L->H, L->Is, L->wdtype, &P->slay) != MOE_OK)
    return MOE_ERR_INVALID_ARG;
  const int rows = T * L->k;
  P->rp = plan_route(T, L->H, L->E, L->k, L->Is > 0 && L->shared_gate_sigmoid);
  P->gu = plan_gemm(gemm_args(P->lay, L->wdtype, true, L->H, L->I, L->E, rows, T));
  P->dn = plan_gemm(gemm_args(P->lay, L->wdtype, false, L->I, L->H, L->E, rows, T));
  if (L->Is) {
    GemmArgs sgu = gemm_args(P->slay, L->wdtype, true, L->H, L->Is, 1, T);
    GemmArgs sdn = gemm_args(P->slay, L->wdtype, false, L->Is, L->H, 1, T);
    P->sgu = plan_gemm(sgu);
    P->sdn = plan_gemm(sdn);
    // the shared expert follows the routed experts' kernel choice, so the two share launches
    if (P->gu.use_tc && P->dn.use_tc && tc_supported(sgu) && tc_supported(sdn)) {
      P->sgu.use_tc = 1;
      P->sdn.use_tc = 1;
    }
    P->merged = P->gu.use_tc && P->dn.use_tc && P->sgu.use_tc && P->sdn.use_tc;
    if (P->merged) {
      P->mgu = plan_tc_pair(gemm_args(P->lay, L->wdtype, true, L->H, L->I, L->E, rows, T), sgu);
      P->mdn = plan_tc_pair(gemm_args(P->lay, L->wdtype, false, L->I, L->H, L->E, rows, T), sdn);
    }
  }
  P->dec = plan_decode(T, L->H, L->E, L->k, L->I, L->Is, L->wdtype,
                       L->Is > 0 && L->shared_gate_sigmoid);
  return MOE_OK;
}

static size_t carve(WsCursor& c, const moe_layer* L, int T, const LayerPlan& P, LayerScratch* s) {
  LayerScratch z{};
  const size_t tk = (size_t)T * L->k;
  // control block, zeroed by one memset per forward: error word and split-K counters (every
  // launch leaves the counters it used at zero again)
  z.err = c.take<int32_t>(64);
  size_t ce = std::max({P.gu.counter_elems, P.dn.counter_elems, P.sgu.counter_elems,
                        P.sdn.counter_elems, P.mgu.t1.counter_elems, P.mdn.t1.counter_elems,
                        P.dec.ok ? P.dec.ctl_words : (size_t)1, (size_t)1});
  z.counters = c.take<int32_t>(ce);
  z.ctl_bytes = c.used;
  route_scratch(c, P.rp, T, L->E, &z.rs);
  z.ids = c.take<int32_t>(tk + 1);
  z.w = c.take<float>(tk + 1);
  z.counts = c.take<int32_t>(L->E);
  z.offsets = c.take<int32_t>(L->E + 1);
  z.pos = c.take<int32_t>(tk + 1);
  z.src = c.take<int32_t>(tk + 1);
  z.tie = c.take<int32_t>(T + 1);
  z.shared_gate = c.take<float>(T + 1);
  z.x_perm = c.take<uint16_t>(tk * L->H + 8);
  z.h = c.take<uint16_t>(tk * L->I + 8);
  z.y_perm = c.take<uint16_t>(tk * L->H + 8);
  if (L->Is) {
    z.h_s = c.take<uint16_t>((size_t)T * L->Is + 8);
    z.s = c.take<uint16_t>((size_t)T * L->H + 8);
  }
  size_t pe = std::max({P.gu.part_elems, P.dn.part_elems, P.sgu.part_elems, P.sdn.part_elems,
                        P.mgu.t1.part_elems, P.mdn.t1.part_elems, (size_t)1});
  z.part = c.take<float>(pe);
  z.part_s = c.take<float>(std::max({P.mgu.t2.part_elems, P.mdn.t2.part_elems, (size_t)1}));
  if (P.dec.ok) {
    z.dec_rpart = c.take<float>((size_t)P.dec.S * T * P.dec.Cp);
    z.dec_gpart = c.take<float>(P.dec.gpart_elems);
    z.dec_dpart = c.take<float>(P.dec.dpart_elems);
    z.dec_ss = c.take<float>((size_t)P.dec.NB * T + 1);
    if (!L->Is) {   // the decode kernel's shared-expert buffers are never read without one
      z.h_s = nullptr;
      z.s = nullptr;
    }
  }
  if (s) *s = z;
  return c.used;
}

// Device-side expert list and bundle table that replace the routing's list (device LRU).
struct DevExperts {
  const int32_t* active = nullptr;
  const int32_t* n_active = nullptr;
  const void* const* tab = nullptr;
};

static int run_experts(const moe_layer* L, const LayerPlan& P, const LayerScratch& s,
                       const BundleTable& tab, int T, int host_n, const int32_t* host_ids,
                       cudaStream_t st, std::function<int()> between,
                       const DevExperts& dx = DevExperts()) {
  const int rows = T * L->k;
  const int32_t* act = dx.active ? dx.active : s.rs.active;
  const int32_t* nact = dx.active ? dx.n_active : s.rs.n_active;
  GemmArgs gu = gemm_args(P.lay, L->wdtype, true, L->H, L->I, L->E, rows, T);
  gu.xin = s.x_perm; gu.offsets = s.offsets; gu.active = act;
  gu.n_active = nact; gu.tab = &tab; gu.out = s.h; gu.dev_tab = dx.tab;
  gu.host_n = host_n; gu.host_ids = host_ids;
  GemmPlan pg = plan_gemm(gu);
  int r = launch_gemm(gu, pg, s.part, s.counters, s.err, st);
  if (r != MOE_OK) return r;
  if (between && (r = between()) != MOE_OK) return r;
  GemmArgs dn = gemm_args(P.lay, L->wdtype, false, L->I, L->H, L->E, rows, T);
  dn.xin = s.h; dn.offsets = s.offsets; dn.active = act;
  dn.n_active = nact; dn.tab = &tab; dn.out = s.y_perm; dn.dev_tab = dx.tab;
  dn.host_n = host_n; dn.host_ids = host_ids;
  GemmPlan pd = plan_gemm(dn);
  return launch_gemm(dn, pd, s.part, s.counters, s.err, st);
}

// Routed experts and the shared expert in one tcgen05 launch per GEMM (the shared expert is the
// extra group: its rows are the T token rows of x, its output h_s / s).
static int run_ffn_merged(const moe_layer* L, const LayerPlan& P, const LayerScratch& s,
                          const BundleTable& tab, const uint16_t* x, int T, cudaStream_t st,
                          std::function<int()> between, const DevExperts& dx = DevExperts()) {
  const int rows = T * L->k;
  BundleTable stab{};
  stab.p[0] = L->shared_bundle;
  const int32_t* meta = s.rs.shared_meta;
  const int32_t* act = dx.active ? dx.active : s.rs.active;
  const int32_t* nact = dx.active ? dx.n_active : s.rs.n_active;
  GemmArgs gu = gemm_args(P.lay, L->wdtype, true, L->H, L->I, L->E, rows, T);
  gu.xin = s.x_perm; gu.offsets = s.offsets; gu.active = act;
  gu.n_active = nact; gu.tab = &tab; gu.out = s.h; gu.dev_tab = dx.tab;
  GemmArgs sgu = gemm_args(P.slay, L->wdtype, true, L->H, L->Is, 1, T);
  sgu.xin = x; sgu.offsets = meta; sgu.active = meta + 2; sgu.n_active = meta + 3;
  sgu.tab = &stab; sgu.out = s.h_s;
  int r = launch_tc_pair(gu, sgu, P.mgu, s.part, s.part_s, s.counters, s.err, st);
  if (r != MOE_OK) return r;
  if (between && (r = between()) != MOE_OK) return r;
  GemmArgs dn = gemm_args(P.lay, L->wdtype, false, L->I, L->H, L->E, rows, T);
  dn.xin = s.h; dn.offsets = s.offsets; dn.active = act;
  dn.n_active = nact; dn.tab = &tab; dn.out = s.y_perm; dn.dev_tab = dx.tab;
  GemmArgs sdn = gemm_args(P.slay, L->wdtype, false, L->Is, L->H, 1, T);
  sdn.xin = s.h_s; sdn.offsets = meta; sdn.active = meta + 2; sdn.n_active = meta + 3;
  sdn.tab = &stab; sdn.out = s.s;
  return launch_tc_pair(dn, sdn, P.mdn, s.part, s.part_s, s.counters, s.err, st);
}

static int run_shared(const moe_layer* L, const LayerPlan& P, const LayerScratch& s,
                      const uint16_t* x, int T, cudaStream_t st) {
  if (!L->Is) return MOE_OK;
  BundleTable tab{};
  tab.p[0] = L->shared_bundle;
  const int32_t* meta = s.rs.shared_meta;
  GemmArgs gu = gemm_args(P.slay, L->wdtype, true, L->H, L->Is, 1, T);
  gu.xin = x; gu.offsets = meta; gu.active = meta + 2; gu.n_active = meta + 3;
  gu.tab = &tab; gu.out = s.h_s;
  int r = launch_gemm(gu, P.sgu, s.part, s.counters, s.err, st);
  if (r != MOE_OK) return r;
  GemmArgs dn = gemm_args(P.slay, L->wdtype, false, L->Is, L->H, 1, T);
  dn.xin = s.h_s; dn.offsets = meta; dn.active = meta + 2; dn.n_active = meta + 3;
  dn.tab = &tab; dn.out = s.s;
  return launch_gemm(dn, P.sdn, s.part, s.counters, s.err, st);
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_last_cuda_error(void) { return g_last_cuda; }

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_CAPACITY: return "MOE_ERR_CAPACITY";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_CORRUPT: return "MOE_ERR_CORRUPT";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_NO_MEMORY: return "MOE_ERR_NO_MEMORY";
    default: return "MOE_ERR_UNKNOWN";
  }
}

int moe_version(void) { return (1 << 16) | 0; }

int moe_set_option(int option, int value) {
  if (option == MOE_OPT_FFN_KERNEL) {
    if (value < 0 || value > 2) return MOE_ERR_INVALID_ARG;
    g_ffn_path = value;
    return MOE_OK;
  }
  if (option == MOE_OPT_DECODE_KERNEL) {
    if (value < 0 || value > 2) return MOE_ERR_INVALID_ARG;
    g_decode_path = value;
    return MOE_OK;
  }
  if (option == MOE_OPT_PDL) {
    if (value < 0 || value > 1) return MOE_ERR_INVALID_ARG;
    g_use_pdl = value;
    return MOE_OK;
  }
  return MOE_ERR_INVALID_ARG;
}

int moe_workspace_error(const void* ws, int32_t* code, void* stream) {
  if (!ws || !code) return MOE_ERR_INVALID_ARG;
  MOE_CUDA_TRY(cudaMemcpyAsync(code, ws, sizeof(int32_t), cudaMemcpyDeviceToHost,
                               (cudaStream_t)stream));
  MOE_CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));
  return MOE_OK;
}

size_t moe_route_workspace_size(int T, int H, int E, int k) {
  if (!valid_route_shape(T, H, E, k)) return 0;
  // the slice count depends on whether the shared-expert gate column is present: size for both
  WsCursor a(nullptr, 0), b(nullptr, 0);
  a.take<int32_t>(64);
  b.take<int32_t>(64);
  return std::max(route_scratch(a, plan_route(T, H, E, k, true), T, E, nullptr),
                  route_scratch(b, plan_route(T, H, E, k, false), T, E, nullptr));
}

int moe_route_topk(const uint16_t* x, const float* w_r, const float* logit_bias,
                   const float* sel_bias, const uint16_t* w_gate, const int32_t* forced_ids,
                   int T, int H, int E, int k, int gating, float scale, int32_t* ids, float* w,
                   int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* src,
                   float* logits, float* shared_gate, int32_t* tie_flags, void* ws,
                   size_t ws_bytes, void* stream) {
  MOE_REQUIRE(valid_route_shape(T, H, E, k));
  MOE_REQUIRE(gating >= 0 && gating <= 2);
  MOE_REQUIRE(counts && offsets && ws);
  MOE_REQUIRE(T == 0 || (x && w_r && ids && w && pos && src));
  MOE_REQUIRE(!w_gate || shared_gate);
  const RoutePlan rp = plan_route(T, H, E, k, w_gate != nullptr);
  WsCursor c(ws, ws_bytes);
  int32_t* err = c.take<int32_t>(64);
  RouteScratch s{};
  route_scratch(c, rp, T, E, &s);
  MOE_REQUIRE(c.ok());
  // the error word (first 4 bytes of ws) starts every call at zero; only the tensor-core
  // router's bounded waits (T >= 256) can set it
  MOE_CUDA_TRY(cudaMemsetAsync(err, 0, sizeof(int32_t), (cudaStream_t)stream));
  RouteArgs a{};
  a.x = x; a.w_r = w_r; a.logit_bias = logit_bias; a.sel_bias = sel_bias; a.w_gate = w_gate;
  a.forced = forced_ids; a.T = T; a.H = H; a.E = E; a.k = k; a.gating = gating;
  a.scale = scale; a.ids = ids; a.counts = counts; a.offsets = offsets; a.pos = pos;
  a.src = src; a.tie_flags = tie_flags; a.w = w; a.logits = logits;
  a.shared_gate = shared_gate; a.x_perm = nullptr; a.err = err;
  return launch_route(a, rp, s, (cudaStream_t)stream);
}

int moe_permute(const uint16_t* x, const int32_t* src, int T, int k, int H, uint16_t* x_perm,
                void* stream) {
  MOE_REQUIRE(T >= 0 && k >= 1 && H > 0 && H % 8 == 0);
  if (T == 0) return MOE_OK;
  MOE_REQUIRE(x && src && x_perm && aligned16(x) && aligned16(x_perm));
  return launch_gather(x, src, T * k, k, H, x_perm, (cudaStream_t)stream);
}

size_t moe_grouped_swiglu_workspace_size(int max_rows, int E, int H, int I, int wdtype) {
  moe_bundle_layout lay;
  if (max_rows < 0 || E <= 0 || E > kMaxExperts || moe_bundle_layout_of(H, I, wdtype, &lay))
    return 0;
  WsCursor c(nullptr, 0);
  c.take<int32_t>(64);
  GemmPlan a = plan_gemm(gemm_args(lay, wdtype, true, H, I, E, max_rows));
  GemmPlan b = plan_gemm(gemm_args(lay, wdtype, false, I, H, E, max_rows));
  c.take<int32_t>(std::max({a.counter_elems, b.counter_elems, (size_t)1}));
  c.take<uint16_t>((size_t)max_rows * I + 8);
  c.take<int32_t>(kMaxExperts + 32);
  c.take<float>(std::max({a.part_elems, b.part_elems, (size_t)1}));
  return c.used;
}

// experts that receive rows, computed on the device from offsets (standalone grouped call)
__global__ void active_from_offsets_kernel(const int32_t* offsets, int E, int32_t* active,
                                           int32_t* n_active) {
  if (threadIdx.x != 0) return;
  int n = 0;
  for (int e = 0; e < E; ++e)
    if (offsets[e + 1] > offsets[e]) active[n++] = e;
  *n_active = n;
}

int moe_grouped_swiglu(const uint16_t* x_perm, const int32_t* offsets,
                       const void* const* bundles, int E, int H, int I, int wdtype,
                       int max_rows, uint16_t* y_perm, void* ws, size_t ws_bytes,
                       void* stream) {
  moe_bundle_layout lay;
  MOE_REQUIRE(E > 0 && E <= kMaxExperts && max_rows >= 0);
  MOE_REQUIRE(moe_bundle_layout_of(H, I, wdtype, &lay) == MOE_OK);
  if (max_rows == 0) return MOE_OK;
  MOE_REQUIRE(x_perm && offsets && bundles && y_perm && ws);
  MOE_REQUIRE(aligned16(x_perm) && aligned16(y_perm));
  cudaStream_t st = (cudaStream_t)stream;
  BundleTable tab{};
  for (int e = 0; e < E; ++e) tab.p[e] = bundles[e];
  WsCursor c(ws, ws_bytes);
  GemmArgs gu = gemm_args(lay, wdtype, true, H, I, E, max_rows);
  GemmArgs dn = gemm_args(lay, wdtype, false, I, H, E, max_rows);
  GemmPlan pg = plan_gemm(gu), pd = plan_gemm(dn);
  // error word and split-K counters first: one memset zeroes both
  int32_t* err = c.take<int32_t>(64);
  int32_t* ctr = c.take<int32_t>(std::max({pg.counter_elems, pd.counter_elems, (size_t)1}));
  const size_t ctl_bytes = c.used;
  uint16_t* h = c.take<uint16_t>((size_t)max_rows * I + 8);
  int32_t* act = c.take<int32_t>(kMaxExperts + 32);
  float* part = c.take<float>(std::max({pg.part_elems, pd.part_elems, (size_t)1}));
  MOE_REQUIRE(c.ok());
  MOE_CUDA_TRY(cudaMemsetAsync(err, 0, ctl_bytes, st));
  active_from_offsets_kernel<<<1, 32, 0, st>>>(offsets, E, act, act + kMaxExperts);
  MOE_COUNT_LAUNCH();
  MOE_LAUNCH_CHECK();
  gu.xin = x_perm; gu.offsets = offsets; gu.active = act; gu.n_active = act + kMaxExperts;
  gu.tab = &tab; gu.out = h;
  int r = launch_gemm(gu, pg, part, ctr, err, st);
  if (r != MOE_OK) return r;
  dn.xin = h; dn.offsets = offsets; dn.active = act; dn.n_active = act + kMaxExperts;
  dn.tab = &tab; dn.out = y_perm;
  return launch_gemm(dn, pd, part, ctr, err, st);
}

int moe_combine(const uint16_t* y_perm, const int32_t* pos, const float* w, int T, int k, int H,
                const uint16_t* shared, const float* shared_gate, const uint16_t* residual,
                uint16_t* out, uint16_t* out_normed, float norm_eps, void* stream) {
  MOE_REQUIRE(T >= 0 && k >= 1 && k <= kMaxK && H > 0 && H % 8 == 0);
  MOE_REQUIRE(!out_normed || (H <= kMaxNormH && norm_eps >= 0.f));
  if (T == 0) return MOE_OK;
  MOE_REQUIRE(y_perm && pos && w && out && aligned16(y_perm) && aligned16(out));
  MOE_REQUIRE(!shared || aligned16(shared));
  MOE_REQUIRE(!residual || aligned16(residual));
  MOE_REQUIRE(!out_normed || aligned16(out_normed));
  return launch_combine(y_perm, pos, w, T, k, H, shared, shared_gate, residual, out, out_normed,
                        norm_eps, (cudaStream_t)stream);
}

size_t moe_layer_workspace_size(const moe_layer* L, int T) {
  LayerPlan P{};
  if (make_plan(L, T, &P) != MOE_OK) return 0;
  WsCursor c(nullptr, 0);
  return carve(c, L, T, P, nullptr);
}

int moe_layer_forward(const moe_layer* L, const uint16_t* x, int T, const int32_t* forced_ids,
                      const uint16_t* residual, uint16_t* out, uint16_t* out_normed,
                      moe_expert_cache* cache, moe_layer_stats* st, int32_t* ids_out,
                      float* w_out, void* ws, size_t ws_bytes, void* stream) {
  LayerPlan P{};
  int r = make_plan(L, T, &P);
  if (r != MOE_OK) return r;
  MOE_REQUIRE(L->gating >= 0 && L->gating <= 2 && L->w_r && ws);
  MOE_REQUIRE(!L->Is || L->shared_bundle);
  MOE_REQUIRE(!(L->Is && L->shared_gate_sigmoid) || L->w_gate);
  MOE_REQUIRE(cache || L->bundles);
  MOE_REQUIRE(!cache || (cache_live(cache) && cache->E == L->E && L->layer_index >= 0 &&
                         L->layer_index < cache->L &&
                         cache->slot_bytes >= P.lay.total_bytes));
  void* const* pev = st ? st->phase_events : nullptr;
  if (st) {
    std::memset(st, 0, sizeof(*st));
    st->phase_events = pev;
  }
  const long long launches0 = g_launches;
  auto phase = [&](int i) -> int {
    if (pev && pev[i]) {
      // inside a stream capture an ordinary record only orders the graph; an external record
      // makes the event fire on every replay of the caller's graph
      cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
      cudaError_t e = cudaStreamIsCapturing((cudaStream_t)stream, &cs);
      if (e != cudaSuccess) return fail_cuda(e);
      e = cs == cudaStreamCaptureStatusActive
              ? cudaEventRecordWithFlags((cudaEvent_t)pev[i], (cudaStream_t)stream,
                                         cudaEventRecordExternal)
              : cudaEventRecord((cudaEvent_t)pev[i], (cudaStream_t)stream);
      if (e != cudaSuccess) return fail_cuda(e);
    }
    return MOE_OK;
  };
  if (T == 0) return MOE_OK;
  MOE_REQUIRE(x && out && aligned16(x) && aligned16(out));
  MOE_REQUIRE(ws && reinterpret_cast<uintptr_t>(ws) % 256 == 0);
  MOE_REQUIRE(!out_normed || (aligned16(out_normed) && L->H <= kMaxNormH && L->norm_eps >= 0.f));
  cudaStream_t s0 = (cudaStream_t)stream;
  WsCursor c(ws, ws_bytes);
  LayerScratch s{};
  carve(c, L, T, P, &s);
  MOE_REQUIRE(c.ok());
  MOE_CUDA_TRY(cudaMemsetAsync(s.err, 0, s.ctl_bytes, s0));

  if ((r = phase(0)) != MOE_OK) return r;
  // (the fused kernel bulk-copies the router slice: W_r and the gate column 16-byte aligned)
  const bool dec_aligned = aligned16(L->w_r) && (!L->w_gate || aligned16(L->w_gate)) &&
                           (!residual || aligned16(residual));
  // auto: INT4 weights only up to 4 tokens; above that the in-register dequantisation on the
  // fused kernel's eight consumer warps per SM is slower than the step-by-step kernels'
  const bool dec_wanted =
      g_decode_path == 2 || (g_decode_path == 1 && (L->wdtype != MOE_W_INT4_G128 || T <= 4));
  if (!cache && P.dec.ok && dec_wanted && dec_aligned && (!L->Is || (s.h_s && s.s))) {
    // small batch, every bundle resident: the whole layer in one cooperative launch
    DecodeArgs da{};
    da.x = x; da.residual = residual; da.forced = forced_ids; da.w_r = L->w_r;
    da.logit_bias = L->logit_bias; da.sel_bias = L->sel_bias;
    da.w_gate = (L->Is && L->shared_gate_sigmoid) ? L->w_gate : nullptr;
    da.T = T; da.H = L->H; da.E = L->E; da.k = L->k; da.I = L->I; da.Is = L->Is;
    da.gating = L->gating; da.wdtype = L->wdtype;
    da.shared_sigmoid = (L->Is && L->shared_gate_sigmoid) ? 1 : 0;
    da.scale = L->scale; da.eps = L->norm_eps;
    for (int e = 0; e < L->E; ++e) da.tab.p[e] = L->bundles[e];
    da.shared = L->shared_bundle; da.lay = P.lay; da.slay = P.slay;
    da.out = out; da.out_n = out_normed;
    da.ids = s.ids; da.counts = s.counts; da.offsets = s.offsets; da.pos = s.pos; da.src = s.src;
    da.tie = s.tie; da.active = s.rs.active; da.n_active = s.rs.n_active; da.w = s.w;
    da.shared_gate = s.shared_gate;
    da.part = s.dec_rpart; da.gpart = s.dec_gpart; da.dpart = s.dec_dpart; da.ss = s.dec_ss;
    da.h = s.h; da.y = s.y_perm; da.hs = s.h_s; da.ys = s.s;
    da.ctl = s.counters; da.err = s.err;
    if ((r = launch_decode(da, P.dec, s0)) != MOE_OK) return r;
    for (int i = 1; i < MOE_N_PHASE_EVENTS; ++i)
      if ((r = phase(i)) != MOE_OK) return r;
    if (st) {
      st->fused_decode = 1;
      st->n_launches = (int32_t)(g_launches - launches0);
    }
    if (ids_out)
      MOE_CUDA_TRY(cudaMemcpyAsync(ids_out, s.ids, sizeof(int32_t) * T * L->k,
                                   cudaMemcpyDeviceToDevice, s0));
    if (w_out)
      MOE_CUDA_TRY(cudaMemcpyAsync(w_out, s.w, sizeof(float) * T * L->k,
                                   cudaMemcpyDeviceToDevice, s0));
    return MOE_OK;
  }
  // A1-A4: route, dispatch and gather into expert order
  RouteArgs ra{};
  ra.x = x; ra.w_r = L->w_r; ra.logit_bias = L->logit_bias; ra.sel_bias = L->sel_bias;
  ra.w_gate = (L->Is && L->shared_gate_sigmoid) ? L->w_gate : nullptr;
  ra.forced = forced_ids; ra.T = T; ra.H = L->H; ra.E = L->E; ra.k = L->k;
  ra.gating = L->gating; ra.scale = L->scale; ra.ids = s.ids; ra.counts = s.counts;
  ra.offsets = s.offsets; ra.pos = s.pos; ra.src = s.src; ra.tie_flags = s.tie; ra.w = s.w;
  ra.logits = nullptr; ra.shared_gate = s.shared_gate; ra.x_perm = s.x_perm; ra.err = s.err;
  r = launch_route(ra, P.rp, s.rs, s0);
  if (r != MOE_OK) return r;
  if ((r = phase(1)) != MOE_OK) return r;
  const float* sgate = (L->Is && L->shared_gate_sigmoid) ? s.shared_gate : nullptr;

  if (!cache) {
    BundleTable tab{};
    for (int e = 0; e < L->E; ++e) tab.p[e] = L->bundles[e];
    if (P.merged) {
      // phase 2 (shared expert) is empty: the shared expert runs inside the routed launches
      if (st) st->shared_merged = 1;
      if ((r = phase(2)) != MOE_OK) return r;
      if ((r = run_ffn_merged(L, P, s, tab, x, T, s0,
                              pev ? [&] { return phase(3); } : std::function<int()>())) != MOE_OK)
        return r;
    } else {
      if ((r = run_shared(L, P, s, x, T, s0)) != MOE_OK) return r;
      if ((r = phase(2)) != MOE_OK) return r;
      if ((r = run_experts(L, P, s, tab, T, -1, nullptr, s0,
                           pev ? [&] { return phase(3); } : std::function<int()>())) != MOE_OK)
        return r;
    }
    if ((r = phase(4)) != MOE_OK) return r;
  } else if (cache->device_lru) {
    // A5 on the GPU: the LRU kernel decides hits and misses from the routing counts, the copy
    // kernel brings the misses in on the cache's stream while the shared expert and the hit
    // experts compute; no host round trip
    if ((r = cache_dev_request(cache, L->layer_index, s.counts, s0, s.err)) != MOE_OK) return r;
    BundleTable none{};
    DevExperts hx;
    hx.active = dev_hit_list(cache);
    hx.n_active = dev_n_hit(cache);
    hx.tab = cache->d_ptrs;
    if (P.merged) {
      // the shared expert rides in the hit experts' launches
      if ((r = phase(2)) != MOE_OK) return r;
      if (st) st->shared_merged = 1;
      if ((r = run_ffn_merged(L, P, s, none, x, T, s0, std::function<int()>(), hx)) != MOE_OK)
        return r;
    } else {
      if ((r = run_shared(L, P, s, x, T, s0)) != MOE_OK) return r;
      if ((r = phase(2)) != MOE_OK) return r;
      if ((r = run_experts(L, P, s, none, T, -1, nullptr, s0, std::function<int()>(), hx)) !=
          MOE_OK)
        return r;
    }
    if ((r = phase(3)) != MOE_OK) return r;
    if ((r = cache_dev_wait_copies(cache, s0)) != MOE_OK) return r;
    DevExperts mx = hx;
    mx.active = dev_miss_list(cache);
    mx.n_active = dev_n_miss(cache);
    if ((r = run_experts(L, P, s, none, T, -1, nullptr, s0, std::function<int()>(), mx)) !=
        MOE_OK)
      return r;
    if ((r = phase(4)) != MOE_OK) return r;
  } else {
    // A5: the layer's expert-use mask crosses to the host, the LRU decides, misses are copied
    // on the cache's copy stream while the shared expert and the hit experts compute.
    // The shared expert needs no routed bundle: it is enqueued before the host waits for the
    // read-back, so the GPU computes it during the round trip.
    MOE_CUDA_TRY(cudaMemcpyAsync(cache->host_counts, s.counts, sizeof(int32_t) * L->E,
                                 cudaMemcpyDeviceToHost, s0));
    MOE_CUDA_TRY(cudaEventRecord(cache->d2h, s0));
    if ((r = run_shared(L, P, s, x, T, s0)) != MOE_OK) return r;
    if ((r = phase(2)) != MOE_OK) return r;
    if ((r = cache_wait_event(cache, cache->d2h)) != MOE_OK) return r;
    uint8_t used[kMaxExperts];
    for (int e = 0; e < L->E; ++e) used[e] = cache->host_counts[e] > 0;
    const void* ptrs[kMaxExperts];
    std::vector<int> hits, misses, waits;
    // from the request on, the layer holds slots: a failure releases them before returning
    // (the release follows whatever this call already enqueued on s0)
    auto fail_released = [&](int code) {
      cache_release(cache, L->layer_index, s0);
      return code;
    };
    r = cache_request_split(cache, L->layer_index, used, s0, ptrs, &hits, &misses, &waits);
    if (r != MOE_OK) return fail_released(r);
    // hits on bundles a prefetch copied: wait for those copies (usually long done)
    for (int slot : waits) {
      const cudaError_t we = cudaStreamWaitEvent(s0, cache->ready[slot], 0);
      if (we != cudaSuccess) return fail_released(fail_cuda(we));
      cache->slot_pending[slot] = 0;
    }
    BundleTable tab{};
    for (int e = 0; e < L->E; ++e) tab.p[e] = ptrs[e];
    if (!hits.empty() && (r = run_experts(L, P, s, tab, T, (int)hits.size(), hits.data(), s0,
                                          std::function<int()>())) != MOE_OK)
      return fail_released(r);
    if ((r = phase(3)) != MOE_OK) return fail_released(r);
    if (!misses.empty()) {
      const cudaError_t we = cudaStreamWaitEvent(s0, cache->last_copy, 0);
      if (we != cudaSuccess) return fail_released(fail_cuda(we));
      if ((r = run_experts(L, P, s, tab, T, (int)misses.size(), misses.data(), s0,
                           std::function<int()>())) != MOE_OK)
        return fail_released(r);
    }
    if ((r = phase(4)) != MOE_OK) return fail_released(r);
    if (st) {
      st->n_unique = (int32_t)(hits.size() + misses.size());
      st->n_missed = (int32_t)misses.size();
    }
  }
  // A9
  r = launch_combine(s.y_perm, s.pos, s.w, T, L->k, L->H, L->Is ? s.s : nullptr, sgate,
                     residual, out, out_normed, L->norm_eps, s0);
  if (r != MOE_OK) {
    if (cache && !cache->device_lru) cache_release(cache, L->layer_index, s0);
    return r;
  }
  if ((r = phase(5)) != MOE_OK) return r;
  if (st) st->n_launches = (int32_t)(g_launches - launches0);
  if (cache && !cache->device_lru) {
    if ((r = cache_release(cache, L->layer_index, s0)) != MOE_OK) return r;
    // lookahead: copy the next layer's predicted experts while this layer still computes
    // (after the last-use record above, so a prefetch that evicts one of this layer's slots
    // waits for this layer)
    if (cache->prefetch_next &&
        (r = cache_prefetch(cache, (L->layer_index + 1) % cache->L, nullptr, nullptr)) != MOE_OK)
      return r;
  }
  if (ids_out)
    MOE_CUDA_TRY(cudaMemcpyAsync(ids_out, s.ids, sizeof(int32_t) * T * L->k,
                                 cudaMemcpyDeviceToDevice, s0));
  if (w_out)
    MOE_CUDA_TRY(cudaMemcpyAsync(w_out, s.w, sizeof(float) * T * L->k,
                                 cudaMemcpyDeviceToDevice, s0));
  return MOE_OK;
}

}  // extern "C"

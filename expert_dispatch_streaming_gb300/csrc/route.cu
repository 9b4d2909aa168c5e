// Routing: router logits (A1), top-k gating (A2), histogram + scan + stable rank (A3) and
// the token gather into expert-contiguous order (A4).
//
// The router picks a handful of experts per token and only those experts run ("NovaLLM:
// Running Massive MoE Models Fully In-Memory", section "2. Why MoE Is a Natural Breakthrough
// Point"); work is then grouped by expert so a batch touches each selected expert once
// (section "3. Optimization #1 -- Expert-Level Streaming").
//
// Kernels
//   router_partial_kernel  fp32 logits of a (token tile, column tile, H slice); the H slices
//                          let a small batch spread the router read over every SM.
//   gate_cta_kernel        one CTA per token (grid-stride): sums the token's slices in fixed
//                          order, scores, ranks the experts over the CTA (gate_token_cta),
//                          re-scores the experts whose fp32 score is within the error margin of
//                          the k-th (the whole CTA, compensated sums), writes ids / weights and
//                          bumps the per-tile expert histogram.
//   gate_topk_kernel       the same gating by one warp per token (gate_token, 1-8 expert slots
//                          per lane), for the largest batches, where throughput rather than one
//                          token's latency counts, and for a few dozen experts from 256 tokens.
//   scan_kernel            one CTA: per-expert counts, exclusive offsets, per-tile bases and
//                          the list of experts that received rows.
//   rank_permute_kernel    one CTA per 128-token tile: stable rank of each (t, j) within its
//                          expert from per-expert token bitmasks, pos / src, and (optionally)
//                          the row copy x -> x_perm with 16-byte vector loads and stores.
//   route_tail_kernel      for a batch of at most kSmallT tokens (decode), everything after
//                          the router product in one CTA: two launches route the batch.
#include "common.cuh"
#include "gate.cuh"
#include "route.cuh"
#include "tc_gemm.cuh"

namespace moe {


// ------------------------------------------------------------------------------ A1 router
constexpr int R_BT = 32, R_KH = 32;
// Column tile of the router product: 64 columns, or 16 for at most 16 (a handful of experts,
// whose 64-column tiles would leave three quarters of the threads without a column).  (With 8
// experts the tensor-core product stays the faster one from 256 tokens on: measured at 4096
// tokens, 60 against 110 us for the whole routing step.)
constexpr int kRouterSmallC = 16;

template <int R_BC>
__global__ void __launch_bounds__(256)
router_partial_kernel(const uint16_t* __restrict__ x, const float* __restrict__ w_r,
                      const uint16_t* __restrict__ w_gate, int T, int H, int E, int C,
                      int h_per_split, float* __restrict__ part, int32_t* __restrict__ hist,
                      int hist_n) {
  pdl_trigger();
  pdl_wait();
  __shared__ float xs[R_KH][R_BT + 1];
  __shared__ float wsm[R_KH][R_BC];
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int t0 = blockIdx.x * R_BT, c0 = blockIdx.y * R_BC, split = blockIdx.z;
  const int h_lo = split * h_per_split, h_hi = min(H, h_lo + h_per_split);

  // the first CTA clears the per-tile histogram the gating kernel accumulates into
  if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
    for (int i = tid; i < hist_n; i += blockDim.x) hist[i] = 0;

  // The loads of up to kPf 32-row tiles are issued together, into registers, before any of
  // them is used: a CTA's slice of a small batch is a few tiles, and one memory latency per
  // tile (load, barrier, compute, barrier) would dominate it.
  constexpr int kPf = 4;
  float xv[kPf][R_BT * R_KH / 256], wv[kPf][R_KH * R_BC / 256];
  auto load = [&](int h0, float (&xq)[R_BT * R_KH / 256], float (&wq)[R_KH * R_BC / 256]) {
    // x tile: 32 tokens x 32 h (bf16 -> fp32); weight tile: 32 h x 64 columns, column E the
    // shared-expert gate vector
#pragma unroll
    for (int j = 0; j < R_BT * R_KH / 256; ++j) {
      const int i = tid + 256 * j, tt = i / R_KH, hh = i % R_KH, t = t0 + tt, h = h0 + hh;
      xq[j] = (t < T && h < h_hi) ? bf16_bits_to_float(x[(size_t)t * H + h]) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < R_KH * R_BC / 256; ++j) {
      const int i = tid + 256 * j, hh = i / R_BC, cc = i % R_BC, h = h0 + hh, c = c0 + cc;
      float v = 0.f;
      if (h < h_hi) {
        if (c < E) v = w_r[(size_t)h * E + c];
        else if (c < C) v = bf16_bits_to_float(w_gate[h]);
      }
      wq[j] = v;
    }
  };
  constexpr int NQ = R_BC / 16;   // columns per thread
  float acc[2][NQ] = {};
  for (int hb = h_lo; hb < h_hi; hb += kPf * R_KH) {
#pragma unroll
    for (int f = 0; f < kPf; ++f)
      if (hb + f * R_KH < h_hi) load(hb + f * R_KH, xv[f], wv[f]);
#pragma unroll
    for (int f = 0; f < kPf; ++f) {
      if (hb + f * R_KH >= h_hi) break;
#pragma unroll
      for (int j = 0; j < R_BT * R_KH / 256; ++j) {
        const int i = tid + 256 * j;
        xs[i % R_KH][i / R_KH] = xv[f][j];
      }
#pragma unroll
      for (int j = 0; j < R_KH * R_BC / 256; ++j) {
        const int i = tid + 256 * j;
        wsm[i / R_BC][i % R_BC] = wv[f][j];
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < R_KH; ++kk) {
        float a0 = xs[kk][ty], a1 = xs[kk][ty + 16];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          float b = wsm[kk][tx + 16 * q];
          acc[0][q] = fmaf(a0, b, acc[0][q]);
          acc[1][q] = fmaf(a1, b, acc[1][q]);
        }
      }
      __syncthreads();
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    int t = t0 + ty + 16 * i;
    if (t >= T) continue;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      int c = c0 + tx + 16 * q;
      if (c < C) part[((size_t)split * T + t) * C + c] = acc[i][q];
    }
  }
}

// Sums the S H-slice partials of every logit into slice 0, in place: eight lanes per logit,
// lane j summing slices j, j + 8, ... in order, the eight sums then combined pairwise by
// shuffles (a fixed order).  Used when a small batch was spread over many slices, so that the
// gate kernel reads one value per logit instead of S.
__global__ void __launch_bounds__(256)
reduce_slices_kernel(float* __restrict__ part, int S, int n) {
  pdl_trigger();
  pdl_wait();
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  const int i = g >> 3, j = g & 7;
  float a = 0.f;
  if (i < n) {
#pragma unroll 4
    for (int sp = j; sp < S; sp += 8) a += part[(size_t)sp * n + i];
  }
  a += __shfl_xor_sync(0xffffffffu, a, 1);
  a += __shfl_xor_sync(0xffffffffu, a, 2);
  a += __shfl_xor_sync(0xffffffffu, a, 4);
  if (i < n && j == 0) part[i] = a;
}

// Tensor-core router input: the router (and shared-expert gate vector as row E) split into three
// bf16 pieces hi + mid + lo (each the bf16 rounding of what the previous pieces leave), which
// represent the fp32 weight; written as a tiled 128-byte-swizzled bf16 image of [Mpad x 3H]
// (piece p of row m at k-tile p * H/64 + k/64), plus the transposed fp32 router for the exact
// re-scoring.  Block = 64 rows m x 64 k: the fp32 router block is read row by row (coalesced)
// into shared memory, then thread (row m, 8-element chunk c of the 64 k), c fastest, writes
// its 16 bytes of each piece's image row -- eight threads one whole 128-byte row -- and its 32
// bytes of the transposed copy (eight threads one 256-byte run).  Block (0, 0) also clears the
// histogram and writes the one-group dispatch {0, T, 0, 1} the router GEMM runs over.
constexpr int kPrepM = 64, kPrepK = 64;
__global__ void __launch_bounds__(256)
router_prep_kernel(const float* __restrict__ w_r, const uint16_t* __restrict__ w_gate, int H,
                   int E, int Mpad, int T, uint16_t* __restrict__ img, float* __restrict__ w_rT,
                   int32_t* __restrict__ hist, int hist_n, int32_t* __restrict__ meta) {
  pdl_trigger();
  pdl_wait();
  __shared__ float blk[kPrepK][kPrepM + 1];
  const int tid = threadIdx.x, m0 = blockIdx.x * kPrepM, h0 = blockIdx.y * kPrepK;
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    for (int i = tid; i < hist_n; i += blockDim.x) hist[i] = 0;
    if (tid == 0) { meta[0] = 0; meta[1] = T; meta[2] = 0; meta[3] = 1; }
  }
  // all 16 loads of a thread issued before the first use (one memory latency, not sixteen)
  float ld[kPrepK * kPrepM / 256];
#pragma unroll
  for (int j = 0; j < kPrepK * kPrepM / 256; ++j) {
    const int i = tid + 256 * j, hh = i / kPrepM, mm = i % kPrepM, m = m0 + mm, h = h0 + hh;
    ld[j] = m < E ? w_r[(size_t)h * E + m]
                  : (m == E && w_gate ? bf16_bits_to_float(w_gate[h]) : 0.f);
  }
#pragma unroll
  for (int j = 0; j < kPrepK * kPrepM / 256; ++j) {
    const int i = tid + 256 * j;
    blk[i / kPrepM][i % kPrepM] = ld[j];
  }
  __syncthreads();
  const int KTB = H / 64, kt = h0 / 64;
#pragma unroll
  for (int i = tid; i < kPrepM * 8; i += 256) {
    const int c = i & 7, mm = i >> 3, m = m0 + mm, mt = m >> 7, r = m & 127;
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = blk[8 * c + j][mm];
    uint32_t pc[3][4];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      float a = v[j], b = v[j + 1];
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const uint32_t w = float2_to_bf16x2(a, b);
        pc[q][j / 2] = w;
        const float2 f = bf16x2_to_float2(w);
        a -= f.x;
        b -= f.y;
      }
    }
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      uint16_t* tile = img + ((size_t)mt * (3 * KTB) + q * KTB + kt) * 8192;
      *reinterpret_cast<uint4*>(tile + r * 64 + ((c ^ (r & 7)) << 3)) =
          make_uint4(pc[q][0], pc[q][1], pc[q][2], pc[q][3]);
    }
    if (m < E && w_rT) {
      float4* o = reinterpret_cast<float4*>(w_rT + (size_t)m * H + h0 + 8 * c);
      o[0] = make_float4(v[0], v[1], v[2], v[3]);
      o[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
}

template <int NC>
__global__ void __launch_bounds__(G_WARPS * 32) gate_topk_kernel(GateParams p) {
  pdl_trigger();
  pdl_wait();
  __shared__ float lrow[G_WARPS][kMaxExperts];
  __shared__ double exact_s[G_WARPS][kMaxExperts];
  const int warp = threadIdx.x >> 5;
  for (int it = 0; it < p.tok_per_warp; ++it) {
    const int t = (blockIdx.x * G_WARPS + warp) * p.tok_per_warp + it;
    if (t >= p.T) break;
    gate_token<NC>(p, t, nullptr, lrow[warp], exact_s[warp]);
  }
}

// A token's gating is a chain of dependent steps (scores, ranks, weights) that one warp runs
// in thousands of serial instructions; spread over a CTA, one thread per expert, it takes a
// few barriers, so a batch's gating time is about that of one token whenever the batch fits
// on the GPU at once (the ranking, weights and tie flags are gate_token's).
constexpr int kGateCtasPerSm = 4;
// Above this many tokens the warp-per-token kernel gates faster (measured with 256 experts at
// 8192 tokens): a CTA waits for its token's rare near-boundary re-scoring with all 8 warps.
constexpr int kGateCtaMaxT = 4096;
// Up to this many experts a warp holds a token's scores in at most two slots per lane and the
// warp-per-token kernel is the faster one from kGateWarpMinT tokens on (measured with 8 and 60
// experts; below, the batch's tokens on as many CTAs finish sooner).
constexpr int kGateWarpMaxE = 64;
constexpr int kGateWarpMinT = 256;
__global__ void __launch_bounds__(kMaxExperts, kGateCtasPerSm) gate_cta_kernel(GateParams p) {
  pdl_trigger();
  pdl_wait();
  __shared__ GateCtaSmem g;
  __shared__ float raw[kMaxExperts + 1];
  __shared__ float lrow0[kMaxExperts];
  __shared__ double exact0[kMaxExperts];
  const int tid = threadIdx.x;
  if (tid < p.E) {
    g.lb[tid] = p.logit_bias ? p.logit_bias[tid] : 0.f;
    g.sb[tid] = p.sel_bias ? p.sel_bias[tid] : 0.f;
  }
  for (int t = blockIdx.x; t < p.T; t += gridDim.x) {
    for (int c = tid; c < p.C; c += kMaxExperts)
      raw[c] = sum_slices(p.part + (size_t)t * p.ldp + c, p.S, (size_t)p.T * p.ldp);
    __syncthreads();
    gate_token_cta<kMaxExperts>(p, t, raw, g, lrow0, exact0, [] { __syncthreads(); });
  }
}

// ------------------------------------------------------------------------------ A3 scan
__global__ void __launch_bounds__(kMaxExperts)
scan_kernel(const int32_t* __restrict__ hist, int ntiles, int E, int32_t* __restrict__ counts,
            int32_t* __restrict__ offsets, int32_t* __restrict__ base,
            int32_t* __restrict__ active, int32_t* __restrict__ n_active,
            int32_t* __restrict__ shared_meta, int T) {
  pdl_trigger();
  pdl_wait();
  __shared__ int s_cnt[kMaxExperts], s_flag[kMaxExperts];
  const int e = threadIdx.x;
  if (shared_meta && e == 0) {
    // a one-group dispatch of all T tokens for the shared expert: offsets {0, T}, active {0}
    shared_meta[0] = 0;
    shared_meta[1] = T;
    shared_meta[2] = 0;
    shared_meta[3] = 1;
  }
  int run = 0;
  if (e < E) {
    for (int tl = 0; tl < ntiles; ++tl) {
      const int c = hist[tl * E + e];
      base[tl * E + e] = run;
      run += c;
    }
  }
  s_cnt[e] = e < E ? run : 0;
  s_flag[e] = (e < E && run > 0) ? 1 : 0;
  __syncthreads();
  // inclusive Hillis-Steele scan of both arrays
  for (int o = 1; o < kMaxExperts; o <<= 1) {
    int a = e >= o ? s_cnt[e - o] : 0;
    int b = e >= o ? s_flag[e - o] : 0;
    __syncthreads();
    s_cnt[e] += a;
    s_flag[e] += b;
    __syncthreads();
  }
  if (e < E) {
    const int excl = s_cnt[e] - run;
    counts[e] = run;
    offsets[e] = excl;
    if (e == E - 1) offsets[E] = s_cnt[e];
    for (int tl = 0; tl < ntiles; ++tl) base[tl * E + e] += excl;
    if (run > 0) active[s_flag[e] - 1] = e;
    if (e == E - 1) *n_active = s_flag[e];
  }
}

// ------------------------------------------------------------------------------ A3+A4
__global__ void __launch_bounds__(256)
rank_permute_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ base, int T,
                    int k, int E, int H, const uint16_t* __restrict__ x,
                    int32_t* __restrict__ pos, int32_t* __restrict__ src,
                    uint16_t* __restrict__ x_perm) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint32_t mask[kMaxExperts][kTileT / 32];
  __shared__ int ptmp[kTileT * kMaxK];
  const int tile = blockIdx.x, t0 = tile * kTileT, tid = threadIdx.x;
  const int ntok = min(kTileT, T - t0);
  for (int i = tid; i < kMaxExperts * (kTileT / 32); i += blockDim.x) (&mask[0][0])[i] = 0u;
  __syncthreads();
  if (tid < ntok)
    for (int j = 0; j < k; ++j) {
      const int e = ids[(size_t)(t0 + tid) * k + j];
      atomicOr(&mask[e][tid >> 5], 1u << (tid & 31));
    }
  __syncthreads();
  if (tid < ntok) {
    const int t = t0 + tid, w = tid >> 5;
    for (int j = 0; j < k; ++j) {
      const int e = ids[(size_t)t * k + j];
      int rank = __popc(mask[e][w] & ((1u << (tid & 31)) - 1u));
      for (int q = 0; q < w; ++q) rank += __popc(mask[e][q]);
      const int pp = base[tile * E + e] + rank;
      pos[(size_t)t * k + j] = pp;
      src[pp] = t * k + j;
      ptmp[tid * k + j] = pp;
    }
  }
  if (x_perm == nullptr) return;
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31, nvec = H / 8;
  for (int q = warp; q < ntok * k; q += blockDim.x / 32) {
    const uint4* s = reinterpret_cast<const uint4*>(x + (size_t)(t0 + q / k) * H);
    uint4* d = reinterpret_cast<uint4*>(x_perm + (size_t)ptmp[q] * H);
    for (int v = lane; v < nvec; v += 32) d[v] = __ldg(s + v);
  }
}

// x_perm[p] = x[src[p] / k]: one warp per destination row
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ src, int rows,
                   int k, int H, uint16_t* __restrict__ x_perm) {
  pdl_trigger();
  pdl_wait();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const int nvec = H / 8;
  const uint4* s = reinterpret_cast<const uint4*>(x + (size_t)(src[warp] / k) * H);
  uint4* d = reinterpret_cast<uint4*>(x_perm + (size_t)warp * H);
#pragma unroll 4
  for (int v = lane; v < nvec; v += 32) d[v] = __ldg(s + v);
}

// x_perm[pos[t k + j]] = x[t] for j < k: one warp per token, each 4 KB piece of the row read
// once and stored to the token's k rows (the destination-order copy above reads every source
// row k times, which the L2 stops absorbing once x_perm's stream evicts x)
__global__ void __launch_bounds__(256)
scatter_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ pos, int T, int k,
                    int H, uint16_t* __restrict__ x_perm) {
  pdl_trigger();
  pdl_wait();
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (t >= T) return;
  const int nvec = H / 8;
  const uint4* s = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  int dst[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) dst[j] = j < k ? __ldg(pos + (size_t)t * k + j) : 0;
  for (int v0 = 0; v0 < nvec; v0 += 256) {
    uint4 q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int v = v0 + lane + 32 * i;
      q[i] = v < nvec ? __ldg(s + v) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j >= k) break;
      uint4* d = reinterpret_cast<uint4*>(x_perm + (size_t)dst[j] * H);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int v = v0 + lane + 32 * i;
        if (v < nvec) d[v] = q[i];
      }
    }
  }
}

// ------------------------------------------------------------------------------ A2-A4, small T
// Everything after the router product for a batch of at most kSmallT tokens, in one CTA (the
// body is route_tail_block in gate.cuh, shared with the fused decode kernel).
constexpr int kTailThreads = 1024;
__global__ void __launch_bounds__(kTailThreads)
route_tail_kernel(GateParams p, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                  int32_t* __restrict__ pos, int32_t* __restrict__ src,
                  int32_t* __restrict__ active, int32_t* __restrict__ n_active,
                  int32_t* __restrict__ shared_meta, uint16_t* __restrict__ x_perm) {
  pdl_trigger();
  pdl_wait();
  __shared__ TailSmem sm;
  route_tail_block<kTailThreads>(p, counts, offsets, pos, src, active, n_active, shared_meta,
                                 x_perm, sm);
}

// ------------------------------------------------------------------------------ host side
RoutePlan plan_route(int T, int H, int E, int k, bool has_gate) {
  RoutePlan r{};
  r.C = E + (has_gate ? 1 : 0);
  r.ntiles = ceil_div(T, kTileT);
  if (T >= kTcRouterMinT && H % 64 == 0) {
    r.tc = 1;
    r.Mpad = (int)round_up(r.C, 128);
    r.S = 1;
    r.h_per_split = H;
    r.tc_S = tc_router_splits(T, H, r.Mpad);
    return r;
  }
  const int tiles = ceil_div(T, R_BT) * ceil_div(r.C, r.C <= kRouterSmallC ? kRouterSmallC : 64);
  const int target = 2 * sm_count();
  // a small batch spreads the router read over the GPU in H slices of as few as 32 rows, so
  // each CTA runs one or two load-compute iterations (the partials are summed by the gate)
  int S = 1;
  if (tiles < target) S = std::min(std::max(1, H / R_KH), ceil_div(target, std::max(tiles, 1)));
  r.h_per_split = round_up(ceil_div(H, S), R_KH);
  r.S = ceil_div(H, r.h_per_split);
  r.small = T >= 1 && T <= kSmallT;   // everything after the router product in one CTA
  return r;
}

size_t route_scratch(WsCursor& c, const RoutePlan& r, int T, int E, RouteScratch* out) {
  RouteScratch s{};
  s.part = c.take<float>((size_t)r.S * T * r.C);
  s.hist = c.take<int32_t>((size_t)std::max(r.ntiles, 1) * E);
  s.base = c.take<int32_t>((size_t)std::max(r.ntiles, 1) * E);
  s.active = c.take<int32_t>(kMaxExperts);
  s.n_active = c.take<int32_t>(32);
  s.shared_meta = c.take<int32_t>(32);
  s.img = nullptr;
  s.w_rT = nullptr;
  s.tc_part = nullptr;
  if (r.tc) {
    s.img = c.take<uint16_t>((size_t)3 * r.Mpad * r.h_per_split);
    s.w_rT = c.take<float>((size_t)E * r.h_per_split);
    if (r.tc_S > 1) {
      s.tc_part = c.take<float>((size_t)r.tc_S * T * r.Mpad);
    }
  }
  if (out) *out = s;
  return c.used;
}

int launch_route(const RouteArgs& a, const RoutePlan& r, const RouteScratch& s,
                 cudaStream_t st) {
  if (a.T > 0) {
    if (r.tc) {
      MOE_LAUNCH_PDL(router_prep_kernel, dim3(r.Mpad / kPrepM, a.H / kPrepK), dim3(256), 0, st,
                     a.w_r, a.w_gate, a.H, a.E, r.Mpad, a.T, s.img, s.w_rT, s.hist,
                     r.ntiles * a.E, s.shared_meta);
      MOE_COUNT_LAUNCH();
      MOE_LAUNCH_CHECK();
      const int rr = launch_tc_router(a.x, a.T, a.H, s.img, r.Mpad, r.C, s.shared_meta, s.part,
                                      s.tc_part, a.err, st);
      if (rr != MOE_OK) return rr;
    } else {
      if (r.C <= kRouterSmallC) {
        dim3 g1(ceil_div(a.T, R_BT), 1, r.S);
        MOE_LAUNCH_PDL(router_partial_kernel<kRouterSmallC>, g1, dim3(256), 0, st, a.x, a.w_r,
                       a.w_gate, a.T, a.H, a.E, r.C, r.h_per_split, s.part, s.hist,
                       r.ntiles * a.E);
      } else {
        dim3 g1(ceil_div(a.T, R_BT), ceil_div(r.C, 64), r.S);
        MOE_LAUNCH_PDL(router_partial_kernel<64>, g1, dim3(256), 0, st, a.x, a.w_r, a.w_gate,
                       a.T, a.H, a.E, r.C, r.h_per_split, s.part, s.hist, r.ntiles * a.E);
      }
      MOE_COUNT_LAUNCH();
      MOE_LAUNCH_CHECK();
    }
    if (r.small) {
      GateParams p{};
      p.part = s.part; p.S = r.S; p.C = r.C; p.ldp = r.C;
      p.x = a.x; p.w_r = a.w_r; p.w_rT = nullptr; p.logit_bias = a.logit_bias;
      p.sel_bias = a.sel_bias; p.forced = a.forced; p.T = a.T; p.H = a.H; p.E = a.E; p.k = a.k;
      p.mode = a.gating; p.scale = a.scale; p.ids = a.ids; p.w = a.w; p.logits = a.logits;
      p.shared_gate = a.shared_gate; p.tie_flags = a.tie_flags; p.hist = nullptr;
      MOE_LAUNCH_PDL(route_tail_kernel, dim3(1), dim3(kTailThreads), 0, st, p, a.counts,
                     a.offsets, a.pos, a.src, s.active, s.n_active, s.shared_meta, a.x_perm);
      MOE_COUNT_LAUNCH();
      MOE_LAUNCH_CHECK();
      return MOE_OK;
    }
    int S_gate = r.S;
    if (r.S > 4) {
      const int n = a.T * r.C;
      MOE_LAUNCH_PDL(reduce_slices_kernel, dim3(ceil_div(8 * n, 256)), dim3(256), 0, st, s.part,
                     r.S, n);
      MOE_COUNT_LAUNCH();
      MOE_LAUNCH_CHECK();
      S_gate = 1;
    }
    GateParams p{};
    p.part = s.part; p.S = S_gate; p.C = r.C; p.ldp = r.C;
    if (r.tc && r.tc_S > 1) {
      // the router GEMM's split partials, [tc_S][T][Mpad]: summed here, in split order
      p.part = s.tc_part;
      p.S = r.tc_S;
      p.ldp = r.Mpad;
    }
    p.x = a.x; p.w_r = a.w_r; p.w_rT = s.w_rT; p.logit_bias = a.logit_bias; p.sel_bias = a.sel_bias;
    p.forced = a.forced; p.T = a.T; p.H = a.H; p.E = a.E; p.k = a.k; p.mode = a.gating;
    p.scale = a.scale; p.ids = a.ids; p.w = a.w; p.logits = a.logits;
    p.shared_gate = a.shared_gate; p.tie_flags = a.tie_flags; p.hist = s.hist;
    if (a.T <= kGateCtaMaxT && (a.E > kGateWarpMaxE || a.T < kGateWarpMinT)) {
      const int ctas = std::min(a.T, kGateCtasPerSm * sm_count());
      MOE_LAUNCH_PDL(gate_cta_kernel, dim3(ctas), dim3(kMaxExperts), 0, st, p);
    } else {
      // one token per warp; four per warp at the largest batches, to amortise the CTA
      p.tok_per_warp = a.T <= 1024 ? 1 : 4;
      const dim3 grid(ceil_div(a.T, G_WARPS * p.tok_per_warp)), block(G_WARPS * 32);
      if (a.E <= 32) MOE_LAUNCH_PDL(gate_topk_kernel<1>, grid, block, 0, st, p);
      else if (a.E <= 64) MOE_LAUNCH_PDL(gate_topk_kernel<2>, grid, block, 0, st, p);
      else if (a.E <= 128) MOE_LAUNCH_PDL(gate_topk_kernel<4>, grid, block, 0, st, p);
      else MOE_LAUNCH_PDL(gate_topk_kernel<EC>, grid, block, 0, st, p);
    }
    MOE_COUNT_LAUNCH();
    MOE_LAUNCH_CHECK();
  }
  MOE_LAUNCH_PDL(scan_kernel, dim3(1), dim3(kMaxExperts), 0, st, s.hist, r.ntiles, a.E,
                 a.counts, a.offsets, s.base, s.active, s.n_active, s.shared_meta, a.T);
  MOE_COUNT_LAUNCH();
  MOE_LAUNCH_CHECK();
  if (a.T > 0) {
    // small batches copy the rows inside the per-tile ranking kernel; large ones gather with
    // one warp per destination row over the whole GPU (the per-tile grid is too small)
    const bool fused_copy =
        a.x_perm && (size_t)a.T * a.k * a.H * 2 <= kFusedGatherMaxBytes && a.T < kSeparateGatherMinT;
    MOE_LAUNCH_PDL(rank_permute_kernel, dim3(r.ntiles), dim3(256), 0, st, a.ids, s.base, a.T,
                   a.k, a.E, a.H, a.x, a.pos, a.src,
                   fused_copy ? a.x_perm : static_cast<uint16_t*>(nullptr));
    MOE_COUNT_LAUNCH();
    MOE_LAUNCH_CHECK();
    if (a.x_perm && !fused_copy) {
      if (a.T >= kSeparateGatherMinT) {
        // large batches: by token (every source row read once)
        MOE_LAUNCH_PDL(scatter_rows_kernel, dim3(ceil_div(a.T * 32, 256)), dim3(256), 0, st,
                       a.x, a.pos, a.T, a.k, a.H, a.x_perm);
        MOE_COUNT_LAUNCH();
        MOE_LAUNCH_CHECK();
      } else {
        // smaller ones: by destination row (k times the warps; x stays in L2)
        const int rr = launch_gather(a.x, a.src, a.T * a.k, a.k, a.H, a.x_perm, st);
        if (rr != MOE_OK) return rr;
      }
    }
  }
  return MOE_OK;
}

int launch_gather(const uint16_t* x, const int32_t* src, int rows, int k, int H,
                  uint16_t* x_perm, cudaStream_t st) {
  if (rows <= 0) return MOE_OK;
  MOE_LAUNCH_PDL(gather_rows_kernel, dim3(ceil_div(rows * 32, 256)), dim3(256), 0, st, x, src,
                 rows, k, H, x_perm);
  MOE_COUNT_LAUNCH();
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe

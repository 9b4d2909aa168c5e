// Gating (A2) and the small-batch routing tail (A2-A4) as device code shared by the routing
// kernels and the fused decode kernel (internal to libmoe).
//
// The router picks a handful of experts per token ("NovaLLM: Running Massive MoE Models Fully
// In-Memory", section "2. Why MoE Is a Natural Breakthrough Point"); the gating formulas are
// those of the workloads' model families (softmax top-k renormalised, softmax over all
// experts, sigmoid with a selection-only bias, renormalised and scaled).
#pragma once
#include <math_constants.h>

#include "common.cuh"
#include "route.cuh"

namespace moe {

// fp32 selection scores within this margin of the k-th are re-scored (exact_score: a
// compensated fp32 dot product, the gating function in fp64).  The fp32
// logit is a sum of H <= 16384 products accumulated in fp32; for the workloads' magnitudes
// its error stays below ~1e-5, so 1e-4 leaves a wide margin (sigmoid scores move by at most
// a quarter of the logit error).
constexpr float kTau = 1e-4f;
constexpr double kNearTie = 1e-6;

// ------------------------------------------------------------------------------ A2 gating
constexpr int G_WARPS = 8;
constexpr int EC = kMaxExperts / 32;  // expert slots per lane

static __device__ __forceinline__ bool better(float sa, int ia, float sb, int ib) {
  return sa > sb || (sa == sb && ia < ib);
}
static __device__ __forceinline__ bool better_d(double sa, int ia, double sb, int ib) {
  return sa > sb || (sa == sb && ia < ib);
}

static __device__ __forceinline__ void warp_argmax(float& s, int& id) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float so = __shfl_xor_sync(0xffffffffu, s, o);
    int io = __shfl_xor_sync(0xffffffffu, id, o);
    if (better(so, io, s, id)) { s = so; id = io; }
  }
}
static __device__ __forceinline__ void warp_argmax_d(double& s, int& id) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    double so = __shfl_xor_sync(0xffffffffu, s, o);
    int io = __shfl_xor_sync(0xffffffffu, id, o);
    if (better_d(so, io, s, id)) { s = so; id = io; }
  }
}
static __device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
static __device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sum of the S H-slice partials of one logit in a fixed order: four interleaved running sums
// (slices s = 0, 4, 8, ... / 1, 5, ... / ...) combined as (a0 + a1) + (a2 + a3), so the loads
// of four slices are in flight together and the result does not depend on scheduling.
static __device__ __forceinline__ float sum_slices(const float* p, int S, size_t stride) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  int sp = 0;
  for (; sp + 4 <= S; sp += 4) {
    a0 += p[(size_t)sp * stride];
    a1 += p[(size_t)(sp + 1) * stride];
    a2 += p[(size_t)(sp + 2) * stride];
    a3 += p[(size_t)(sp + 3) * stride];
  }
  if (sp < S) a0 += p[(size_t)sp * stride];
  if (sp + 1 < S) a1 += p[(size_t)(sp + 1) * stride];
  if (sp + 2 < S) a2 += p[(size_t)(sp + 2) * stride];
  return (a0 + a1) + (a2 + a3);
}

// Error-free transformations in fp32 (no fp64: GB300's fp64 rate is a small fraction of its
// fp32 rate).  Each product x*w of a bf16 and an fp32 is split exactly into p + e (p the fp32
// product, e = fma(x, w, -p)); each addition into a running sum hi is split exactly into the
// new hi and its rounding error (Knuth's TwoSum), and the errors are gathered in lo.  The
// intrinsics keep the compiler from contracting these steps into fused multiply-adds.
static __device__ __forceinline__ void two_sum_into(float& hi, float& lo, float a) {
  const float s = __fadd_rn(hi, a);
  const float bp = __fsub_rn(s, hi);
  const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(a, bp));
  hi = s;
  lo = __fadd_rn(lo, err);
}
static __device__ __forceinline__ void dot_term(float& hi, float& lo, float x, float w) {
  const float p = __fmul_rn(x, w);
  const float e = __fmaf_rn(x, w, -p);
  two_sum_into(hi, lo, p);
  lo = __fadd_rn(lo, e);
}
// (hi, lo) += (hi2, lo2)
static __device__ __forceinline__ void df_add(float& hi, float& lo, float hi2, float lo2) {
  two_sum_into(hi, lo, hi2);
  lo = __fadd_rn(lo, lo2);
}

// Selection score of expert b for token t, accurate to far below the fp32 logit's error (the
// refinement of near-boundary experts): the dot product x . W_r[:, b] in compensated fp32
// (error of order H * 2^-48 * sum |x_h w_h|, about 1e-9 for the workloads' magnitudes against
// the 1e-6 that decides a tie), then the bias and the sigmoid in fp64.
static __device__ __forceinline__ double exact_score(const GateParams& p, int t, int b, int lane) {
  const uint16_t* xr = p.x + (size_t)t * p.H;
  float hi[4] = {0.f, 0.f, 0.f, 0.f}, lo[4] = {0.f, 0.f, 0.f, 0.f};
  if (p.w_rT) {
    // the transposed router row: each lane takes 8 consecutive h per 256 (16-byte loads of x,
    // 32 of W_r), four such chunks in flight before any arithmetic; four sums (fixed order)
    const float* wr = p.w_rT + (size_t)b * p.H;
    const int nch = p.H / 8;                   // 8-element chunks (H is a multiple of 8)
    int c = lane;
    for (; c + 96 < nch; c += 128) {
      uint4 xq[4];
      float4 wa[4], wb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xq[i] = *reinterpret_cast<const uint4*>(xr + 8 * (c + 32 * i));
        wa[i] = *reinterpret_cast<const float4*>(wr + 8 * (c + 32 * i));
        wb[i] = *reinterpret_cast<const float4*>(wr + 8 * (c + 32 * i) + 4);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 x01 = bf16x2_to_float2(xq[i].x), x23 = bf16x2_to_float2(xq[i].y);
        const float2 x45 = bf16x2_to_float2(xq[i].z), x67 = bf16x2_to_float2(xq[i].w);
        dot_term(hi[i], lo[i], x01.x, wa[i].x);
        dot_term(hi[i], lo[i], x01.y, wa[i].y);
        dot_term(hi[i], lo[i], x23.x, wa[i].z);
        dot_term(hi[i], lo[i], x23.y, wa[i].w);
        dot_term(hi[i], lo[i], x45.x, wb[i].x);
        dot_term(hi[i], lo[i], x45.y, wb[i].y);
        dot_term(hi[i], lo[i], x67.x, wb[i].z);
        dot_term(hi[i], lo[i], x67.y, wb[i].w);
      }
    }
    for (; c < nch; c += 32)
      for (int i = 0; i < 8; ++i) dot_term(hi[0], lo[0], bf16_bits_to_float(xr[8 * c + i]), wr[8 * c + i]);
  } else {
    // strided column reads (one row of W_r per lane): eight loads in flight, four sums
    const float* wc = p.w_r + b;
    const size_t E = p.E;
    int h = lane;
    for (; h + 224 < p.H; h += 256) {
      float xv[8], wv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        xv[i] = bf16_bits_to_float(xr[h + 32 * i]);
        wv[i] = wc[(size_t)(h + 32 * i) * E];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) dot_term(hi[i & 3], lo[i & 3], xv[i], wv[i]);
    }
    for (; h < p.H; h += 32) dot_term(hi[0], lo[0], bf16_bits_to_float(xr[h]), wc[(size_t)h * E]);
  }
  df_add(hi[0], lo[0], hi[1], lo[1]);
  df_add(hi[2], lo[2], hi[3], lo[3]);
  df_add(hi[0], lo[0], hi[2], lo[2]);
  // warp sum by a butterfly (lane 0's result is the one the caller keeps: a fixed order)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float h2 = __shfl_xor_sync(0xffffffffu, hi[0], o);
    const float l2 = __shfl_xor_sync(0xffffffffu, lo[0], o);
    df_add(hi[0], lo[0], h2, l2);
  }
  double d = (double)hi[0] + (double)lo[0];
  if (p.logit_bias) d += (double)p.logit_bias[b];
  if (p.mode == MOE_GATING_SIGMOID_BIAS_RENORM) {
    d = 1.0 / (1.0 + exp(-d));
    if (p.sel_bias) d += (double)p.sel_bias[b];
  }
  return d;
}

// exact_score by the NT threads of a CTA: thread i takes the 8-element chunks i, i + NT, ...
// of the dot product (compensated fp32), each warp combines its lanes by the butterfly, and
// thread 0 the warps' pairs in warp order, then adds the bias and the sigmoid in fp64.  For
// the one token whose selection waits on it, the H-long dot product spread over the CTA
// costs about one memory latency instead of one per 256 elements.  `wpart` holds 2 floats
// per warp; all NT threads must call it; `sync` is their barrier; the result is thread 0's.
template <int NT, class Sync>
static __device__ __forceinline__ double exact_score_cta(const GateParams& p, int t, int b,
                                                         float* wpart, Sync sync) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const uint16_t* xr = p.x + (size_t)t * p.H;
  float hi = 0.f, lo = 0.f;
  const int nch = p.H / 8;
  if (p.w_rT) {
    const float* wr = p.w_rT + (size_t)b * p.H;
    for (int c = tid; c < nch; c += NT) {
      const uint4 xq = *reinterpret_cast<const uint4*>(xr + 8 * c);
      const float4 wa = *reinterpret_cast<const float4*>(wr + 8 * c);
      const float4 wb = *reinterpret_cast<const float4*>(wr + 8 * c + 4);
      const float2 x01 = bf16x2_to_float2(xq.x), x23 = bf16x2_to_float2(xq.y);
      const float2 x45 = bf16x2_to_float2(xq.z), x67 = bf16x2_to_float2(xq.w);
      dot_term(hi, lo, x01.x, wa.x);
      dot_term(hi, lo, x01.y, wa.y);
      dot_term(hi, lo, x23.x, wa.z);
      dot_term(hi, lo, x23.y, wa.w);
      dot_term(hi, lo, x45.x, wb.x);
      dot_term(hi, lo, x45.y, wb.y);
      dot_term(hi, lo, x67.x, wb.z);
      dot_term(hi, lo, x67.y, wb.w);
    }
  } else {
    const float* wc = p.w_r + b;
    const size_t E = p.E;
    for (int c = tid; c < nch; c += NT) {
      float xv[8], wv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        xv[i] = bf16_bits_to_float(xr[8 * c + i]);
        wv[i] = wc[(size_t)(8 * c + i) * E];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) dot_term(hi, lo, xv[i], wv[i]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, lo, o);
    df_add(hi, lo, h2, l2);
  }
  if (lane == 0) {
    wpart[2 * w] = hi;
    wpart[2 * w + 1] = lo;
  }
  sync();
  double d = 0.0;
  if (tid == 0) {
    float h = wpart[0], l = wpart[1];
    for (int w2 = 1; w2 < NT / 32; ++w2) df_add(h, l, wpart[2 * w2], wpart[2 * w2 + 1]);
    d = (double)h + (double)l;
    if (p.logit_bias) d += (double)p.logit_bias[b];
    if (p.mode == MOE_GATING_SIGMOID_BIAS_RENORM) {
      d = 1.0 / (1.0 + exp(-d));
      if (p.sel_bias) d += (double)p.sel_bias[b];
    }
  }
  sync();
  return d;
}

// Chosen list (ascending id, or the forced order) and weights of token t by one warp, from the
// lane's logits l[c] (experts lane + 32 c), its chosen flags and the token's logits row lrow.
template <int NC>
static __device__ __forceinline__ void gate_finish(const GateParams& p, int t,
                                                   const float (&l)[NC], const bool (&chosen)[NC],
                                                   const float* lrow, int flag) {
  const int lane = threadIdx.x & 31;
  const int E = p.E, k = p.k;
  {
    // ---- chosen list (ascending id, or the forced order) and weights (lane 0)
    int my_ids[kMaxK];
    if (p.forced) {
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        my_ids[j] = j < k ? min(max(p.forced[(size_t)t * k + j], 0), E - 1) : 0;
    } else {
      int n = 0;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) my_ids[j] = 0;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        unsigned m = __ballot_sync(0xffffffffu, chosen[c]);
        while (m) {
          const int e = 32 * c + __ffs(m) - 1;
          m &= m - 1;
#pragma unroll
          for (int j = 0; j < kMaxK; ++j)
            if (j == n) my_ids[j] = e;
          ++n;
        }
      }
    }

    // softmax over all E needs the warp-wide max and sum
    float M = 0.f, Ssum = 1.f;
    if (p.mode == MOE_GATING_SOFTMAX) {
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int c = 0; c < NC; ++c) mx = fmaxf(mx, l[c]);
      M = warp_max(mx);
      float s = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c)
        if (lane + 32 * c < E) s += expf(l[c] - M);
      Ssum = warp_sum(s);
    }
    __syncwarp();
    if (lane == 0) {
      float v[kMaxK];
      float denom = 0.f, mx = -CUDART_INF_F;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (j < k) mx = fmaxf(mx, lrow[my_ids[j]]);
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        v[j] = 0.f;
        if (j < k) {
          const float lj = lrow[my_ids[j]];
          if (p.mode == MOE_GATING_SOFTMAX_RENORM) v[j] = expf(lj - mx);
          else if (p.mode == MOE_GATING_SOFTMAX) v[j] = expf(lj - M);
          else v[j] = 1.f / (1.f + expf(-lj));
          denom += v[j];
        }
      }
      if (p.mode == MOE_GATING_SOFTMAX) denom = Ssum;
      const float inv = p.scale / denom;
      const int tile = t / kTileT;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < k) {
          p.ids[(size_t)t * k + j] = my_ids[j];
          if (p.ids_local) p.ids_local[j] = my_ids[j];
          p.w[(size_t)t * k + j] = v[j] * inv;
          atomicAdd(&p.hist[tile * E + my_ids[j]], 1);
        }
      }
      if (p.tie_flags) p.tie_flags[t] = flag;
    }
    __syncwarp();
    }
}

// Selection for token t by one warp: scores, top-k with the refinement of near-boundary
// experts by exact_score.  Out: the lane's logits l[c] and chosen flags (experts lane + 32 c), the tie flag;
// writes the token's logits row lrow, logits and shared gate.  `raw` = the token's C summed
// router outputs (or NULL: sum the S slices of p.part); lrow / exact_s = this warp's
// shared-memory rows; pre: exact_s already holds the re-scored band (NaN where not).  NC =
// expert slots per lane (E <= 32 NC): small expert counts run fewer slots' instructions.
// Inlined into each kernel, so that the parameter block's fields and the
// lane arrays stay in registers.
template <int NC>
static __device__ __forceinline__ void gate_select(const GateParams& p, int t, const float* raw,
                                                   float* lrow, double* exact_s, float (&l)[NC],
                                                   bool (&chosen)[NC], int& flag_out,
                                                   bool pre = false) {
  const int lane = threadIdx.x & 31;
  const int E = p.E, k = p.k;
  {
    // ---- logits: fixed-order sum of the H slices (+ logit bias), scores
    float sc[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int e = lane + 32 * c;
      float v = -CUDART_INF_F, s = -CUDART_INF_F;
      if (e < E) {
        v = raw ? raw[e] : sum_slices(p.part + (size_t)t * p.ldp + e, p.S, (size_t)p.T * p.ldp);
        if (p.logit_bias) v += p.logit_bias[e];
        s = v;
        if (p.mode == MOE_GATING_SIGMOID_BIAS_RENORM) {
          s = 1.f / (1.f + expf(-v));
          if (p.sel_bias) s += p.sel_bias[e];
        }
        lrow[e] = v;
        if (p.logits) p.logits[(size_t)t * E + e] = v;
      }
      l[c] = v;
      sc[c] = s;
    }
    if (lane == 0 && p.shared_gate && p.C > E) {
      const float z =
          raw ? raw[E] : sum_slices(p.part + (size_t)t * p.ldp + E, p.S, (size_t)p.T * p.ldp);
      p.shared_gate[t] = 1.f / (1.f + expf(-z));
    }

#pragma unroll
    for (int c = 0; c < NC; ++c) chosen[c] = false;
    int flag = 0;

    if (p.forced == nullptr) {
      // ---- top-(k+1) by repeated warp argmax on (score desc, id asc); kth = the k-th score,
      // nxt = the best unchosen one (scalars, so that nothing here is indexed at run time)
      bool taken[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) taken[c] = (lane + 32 * c) >= E;
      float kth = -CUDART_INF_F, nxt = -CUDART_INF_F;
      const int nsel = min(k + 1, E);
#pragma unroll
      for (int r = 0; r < kMaxK + 1; ++r) {
        if (r < nsel) {
          float bs = -CUDART_INF_F;
          int bi = 0x7fffffff;
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            const int e = lane + 32 * c;
            if (!taken[c] && better(sc[c], e, bs, bi)) { bs = sc[c]; bi = e; }
          }
          warp_argmax(bs, bi);
          if (r == k - 1) kth = bs;
          if (r == k) nxt = bs;
#pragma unroll
          for (int c = 0; c < NC; ++c)
            if (lane + 32 * c == bi) { taken[c] = true; if (r < k) chosen[c] = true; }
        }
      }
      if (k < E && kth - nxt <= kTau) {
        // ---- refinement: experts within the margin of the boundary are re-scored
        // (exact_score); chosen experts clear of it (score - nxt > kTau) stay chosen
        flag = 1;
        bool band[NC];
        int n_def = 0;
        const float thr = kth - kTau;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int e = lane + 32 * c;
          const bool d = chosen[c] && sc[c] - nxt > kTau;
          band[c] = (e < E) && !d && sc[c] >= thr;
          chosen[c] = d;
          n_def += __popc(__ballot_sync(0xffffffffu, d));
        }
        // the band as eight warp-uniform words; one (not unrolled) loop over its members, so
        // that exact_score is inlined once
        unsigned bm[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) bm[c] = __ballot_sync(0xffffffffu, band[c]);
#pragma unroll 1
        for (int c = 0; c < NC; ++c) {
          unsigned m = 0;
#pragma unroll
          for (int c2 = 0; c2 < NC; ++c2) m = c2 == c ? bm[c2] : m;
          while (m) {
            const int b = 32 * c + __ffs(m) - 1;
            m &= m - 1;
            // (pre: the caller re-scored the band already; a NaN marks one it did not)
            double s = pre ? exact_s[b] : CUDART_NAN;
            if (s != s) s = exact_score(p, t, b, lane);
            __syncwarp();
            if (lane == 0) exact_s[b] = s;
          }
        }
        __syncwarp();
        const int need = k - n_def;
        double last = CUDART_INF;
        for (int r = 0; r < need; ++r) {
          double bs = -CUDART_INF;
          int bi = 0x7fffffff;
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            const int e = lane + 32 * c;
            if (band[c] && !chosen[c] && better_d(exact_s[e], e, bs, bi)) {
              bs = exact_s[e];
              bi = e;
            }
          }
          warp_argmax_d(bs, bi);
          last = bs;
#pragma unroll
          for (int c = 0; c < NC; ++c)
            if (lane + 32 * c == bi) chosen[c] = true;
        }
        // exact gap to the best band member left out
        double bs = -CUDART_INF;
        int bi = 0x7fffffff;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int e = lane + 32 * c;
          if (band[c] && !chosen[c] && better_d(exact_s[e], e, bs, bi)) {
            bs = exact_s[e];
            bi = e;
          }
        }
        warp_argmax_d(bs, bi);
        if (bi != 0x7fffffff && last - bs < kNearTie) flag = 2;
      }
    }
    __syncwarp();
    flag_out = flag;
  }
}

// Gating of token t by one warp: gate_select, then the chosen list and weights (gate_finish);
// writes ids / w / logits / shared gate / tie flag of t and adds the token's experts to
// hist[(t / 128) * E + e].
template <int NC = EC>
static __device__ __forceinline__ void gate_token(const GateParams& p, int t, const float* raw,
                                                  float* lrow, double* exact_s) {
  float l[NC];
  bool chosen[NC];
  int flag = 0;
  gate_select<NC>(p, t, raw, lrow, exact_s, l, chosen, flag);
  gate_finish<NC>(p, t, l, chosen, lrow, flag);
}

// ------------------------------------------------------------------------------ A2-A4, small T
// Everything after the router product for a batch of at most kSmallT tokens, by one CTA of NT
// threads: the S slice partials of every logit summed in fixed order (a group of G lanes per
// logit, each lane summing every G-th slice, then a shuffle tree), gating / top-k (one warp per
// token), the expert histogram and scan, the stable ranks and (x_perm not NULL) the row copy
// into expert order.
struct alignas(16) GateCtaSmem {
  float l[kMaxExperts], s[kMaxExperts];   // one token's logits and selection scores
  float lb[kMaxExperts], sb[kMaxExperts]; // logit / selection biases (loaded ahead by the caller)
  int rank[kMaxExperts];
  float cs[8 * (kMaxK + 1)];              // candidates: score, expert
  int ci[8 * (kMaxK + 1)];
  int wc[8];                              // per-warp counts
  float vv[kMaxK];                        // unnormalised weights of the chosen, ascending id
  int vid[kMaxK];
  float kth, nxt;                         // k-th and (k+1)-th selection scores
  float M, Ssum, inv;
  float wpart[16];                        // per-warp (hi, lo) pairs of a re-scoring
  unsigned band[8];                       // per-warp masks of the experts to re-score
};

struct TailSmem {
  float lg[kSmallT * (kMaxExperts + 1)];   // summed router outputs of all tokens
  float lrow[G_WARPS][kMaxExperts];
  double exact_s[G_WARPS][kMaxExperts];
  int hist[kMaxExperts], excl[kMaxExperts], srow[kSmallT * kMaxK];
};

// The fused decode kernel's gating scratch: the routing tail's and gate_token_cta's.
struct CtaGateSmem {
  TailSmem tail;
  GateCtaSmem gc;
};

// Gating of token t by the 256 threads of eight warps (small batches, where one token's gating
// is on the critical path): the same selection rule and the same weights as gate_token, with
// the serial steps spread over the CTA.  Top-(k+1): thread e ranks expert e within its warp's
// 32 (score desc, id asc); the at most k + 1 best of each warp are the candidates, and a
// candidate's rank among the candidates is its rank among all experts whenever that is below
// k + 1 (every expert that beats it beats it in its own warp too, so is a candidate).  The
// weights are computed per chosen expert and normalised by one thread summing them in
// ascending-id order, as gate_finish does.  When ids are forced, or the k-th and (k+1)-th fp32
// scores lie within the margin kTau, the first warp runs gate_select / gate_finish instead
// (with lrow0 / exact0 as that warp's rows; the CTA re-scores the margin's experts first).  raw: the token's C summed
// router outputs (shared memory); g.lb / g.sb hold the biases (zero when absent).  Threads
// 0 .. NT-1 must all call it; `sync` is their barrier.
template <int NT, class Sync>
static __device__ __forceinline__ void gate_token_cta(const GateParams& p, int t, const float* raw,
                                                      GateCtaSmem& g, float* lrow0, double* exact0,
                                                      Sync sync) {
  static_assert(NT == kMaxExperts && NT == 8 * 32, "one thread per expert, eight warps");
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, E = p.E, k = p.k;
  {
    float v = -CUDART_INF_F, sc = -CUDART_INF_F;
    if (tid < E) {
      v = raw[tid] + g.lb[tid];
      sc = v;
      if (p.mode == MOE_GATING_SIGMOID_BIAS_RENORM) sc = 1.f / (1.f + expf(-v)) + g.sb[tid];
      if (p.logits) p.logits[(size_t)t * E + tid] = v;
    }
    g.l[tid] = v;
    g.s[tid] = sc;
    g.rank[tid] = kMaxExperts;
  }
  if (tid == 0 && p.shared_gate && p.C > E) p.shared_gate[t] = 1.f / (1.f + expf(-raw[E]));
  if (tid == 0) g.kth = g.nxt = -CUDART_INF_F;
  sync();
  // ---- candidates: the k + 1 best of each warp's 32 experts
  const int kp = min(k + 1, E);
  const float se = g.s[tid];
  int wr = 0;
  if (w * 32 < E) {
#pragma unroll
    for (int j4 = 0; j4 < 8; ++j4) {
      const float4 s4 = *reinterpret_cast<const float4*>(g.s + w * 32 + 4 * j4);
      const int e0 = w * 32 + 4 * j4;
      wr += better(s4.x, e0, se, tid) + better(s4.y, e0 + 1, se, tid) +
            better(s4.z, e0 + 2, se, tid) + better(s4.w, e0 + 3, se, tid);
    }
  }
  const bool cand = tid < E && wr < kp;
  const unsigned cm = __ballot_sync(0xffffffffu, cand);
  if (lane == 0) g.wc[w] = __popc(cm);
  sync();
  int base = 0, ncand = 0;
#pragma unroll
  for (int w2 = 0; w2 < 8; ++w2) {
    const int c = g.wc[w2];
    base += w2 < w ? c : 0;
    ncand += c;
  }
  if (cand) {
    const int idx = base + __popc(cm & ((1u << lane) - 1u));
    g.cs[idx] = se;
    g.ci[idx] = tid;
  }
  sync();
  // ---- ranks of the candidates among the candidates
  if (tid < ncand) {
    const float sc = g.cs[tid];
    const int id = g.ci[tid];
    int r = 0;
    for (int c = 0; c < ncand; ++c) r += better(g.cs[c], g.ci[c], sc, id);
    g.rank[id] = r;
    if (r == k - 1) g.kth = sc;
    if (r == k) g.nxt = sc;
  }
  sync();
  const bool slow = p.forced != nullptr || (k < E && g.kth - g.nxt <= kTau);
  if (slow) {
    const bool pre = p.forced == nullptr;
    if (pre) {
      // the experts gate_select re-scores (its band: not clear of the boundary by kTau, and
      // within kTau of the k-th score), re-scored here by the whole CTA; gate_select's own
      // fp32 scores and margins are these, so it finds them all (a NaN would make it score a
      // missing one itself)
      const float sc = g.s[tid];
      const bool def = tid < E && g.rank[tid] < k && sc - g.nxt > kTau;
      const bool band = tid < E && !def && sc >= g.kth - kTau;
      exact0[tid] = CUDART_NAN;
      const unsigned bm = __ballot_sync(0xffffffffu, band);
      if (lane == 0) g.band[w] = bm;
      sync();
      for (int w2 = 0; w2 < 8; ++w2) {
        unsigned m = g.band[w2];
        while (m) {
          const int b = 32 * w2 + __ffs(m) - 1;
          m &= m - 1;
          const double d = exact_score_cta<NT>(p, t, b, g.wpart, sync);
          if (tid == 0) exact0[b] = d;
        }
      }
      sync();
    }
    if (tid < 32) {
      float l[EC];
      bool chosen[EC];
      int flag = 0;
      gate_select<EC>(p, t, raw, lrow0, exact0, l, chosen, flag, pre);
      gate_finish<EC>(p, t, l, chosen, g.l, flag);
    }
    sync();
    return;
  }
  // ---- the chosen in ascending id order, their weights
  const bool ch = tid < E && g.rank[tid] < k;
  const unsigned m = __ballot_sync(0xffffffffu, ch);
  if (lane == 0) g.wc[w] = __popc(m);
  if (w == 0 && p.mode == MOE_GATING_SOFTMAX) {
    // softmax over all E: the warp-wide max and sum, in gate_finish's order
    float mx = -CUDART_INF_F;
#pragma unroll
    for (int c = 0; c < EC; ++c) mx = fmaxf(mx, lane + 32 * c < E ? g.l[lane + 32 * c] : -CUDART_INF_F);
    const float Mx = warp_max(mx);
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < EC; ++c)
      if (lane + 32 * c < E) sum += expf(g.l[lane + 32 * c] - Mx);
    sum = warp_sum(sum);
    if (lane == 0) {
      g.M = Mx;
      g.Ssum = sum;
    }
  }
  sync();
  if (ch) {
    int pos = __popc(m & ((1u << lane) - 1u));
#pragma unroll
    for (int w2 = 0; w2 < 8; ++w2) pos += w2 < w ? g.wc[w2] : 0;
    g.vid[pos] = tid;
  }
  sync();
  if (tid < k) {
    const float lj = g.l[g.vid[tid]];
    float v;
    if (p.mode == MOE_GATING_SOFTMAX_RENORM) {
      float mx = -CUDART_INF_F;
      for (int j = 0; j < k; ++j) mx = fmaxf(mx, g.l[g.vid[j]]);
      v = expf(lj - mx);
    } else if (p.mode == MOE_GATING_SOFTMAX) {
      v = expf(lj - g.M);
    } else {
      v = 1.f / (1.f + expf(-lj));
    }
    g.vv[tid] = v;
  }
  sync();
  if (tid == 0) {
    float denom = 0.f;
    for (int j = 0; j < k; ++j) denom += g.vv[j];
    if (p.mode == MOE_GATING_SOFTMAX) denom = g.Ssum;
    g.inv = p.scale / denom;
    if (p.tie_flags) p.tie_flags[t] = 0;
  }
  sync();
  if (tid < k) {
    const int e = g.vid[tid];
    p.ids[(size_t)t * k + tid] = e;
    if (p.ids_local) p.ids_local[tid] = e;
    p.w[(size_t)t * k + tid] = g.vv[tid] * g.inv;
    atomicAdd(&p.hist[(t / kTileT) * E + e], 1);
  }
  sync();
}

// Histogram (already in sm.hist), exclusive scan, list of experts with rows, stable ranks
// (pos / src) and, x_perm not NULL, the row copy into expert order, for the T * k pairs of
// ids, by one CTA of NT threads.
template <int NT>
static __device__ void route_dispatch_block(const int32_t* ids, int T, int k, int E,
                                            int32_t* __restrict__ counts,
                                            int32_t* __restrict__ offsets,
                                            int32_t* __restrict__ pos, int32_t* __restrict__ src,
                                            int32_t* __restrict__ active,
                                            int32_t* __restrict__ n_active,
                                            int32_t* __restrict__ shared_meta,
                                            uint16_t* __restrict__ x_perm,
                                            const uint16_t* __restrict__ x, int H, TailSmem& sm) {
  static_assert(NT >= kMaxExperts, "the scan takes one thread per expert");
  int* hist = sm.hist;
  int* excl = sm.excl;
  int* srow = sm.srow;
  const int tid = threadIdx.x;
  // ---- scan over the experts: counts, exclusive offsets, list of experts with rows
  const bool ex = tid < kMaxExperts;
  int cnt = 0, flag = 0;
  if (ex && tid < E) {
    cnt = hist[tid];
    flag = cnt > 0;
  }
  if (ex) excl[tid] = cnt;
  __syncthreads();
  for (int o = 1; o < kMaxExperts; o <<= 1) {
    const int v = (ex && tid >= o) ? excl[tid - o] : 0;
    __syncthreads();
    if (ex) excl[tid] += v;
    __syncthreads();
  }
  const int incl = ex ? excl[tid] : 0;
  __syncthreads();
  if (ex) {
    excl[tid] = incl - cnt;
    hist[tid] = flag;
  }
  __syncthreads();
  for (int o = 1; o < kMaxExperts; o <<= 1) {
    const int v = (ex && tid >= o) ? hist[tid - o] : 0;
    __syncthreads();
    if (ex) hist[tid] += v;   // inclusive count of experts with rows
    __syncthreads();
  }
  if (tid < E) {
    counts[tid] = cnt;
    offsets[tid] = excl[tid];
    if (tid == E - 1) {
      offsets[E] = excl[tid] + cnt;
      *n_active = hist[tid];
    }
    if (flag) active[hist[tid] - 1] = tid;
  }
  if (tid == 0 && shared_meta) {
    shared_meta[0] = 0;
    shared_meta[1] = T;
    shared_meta[2] = 0;
    shared_meta[3] = 1;
  }
  // ---- stable ranks: pair i = t*k + j goes after every earlier pair routed to its expert
  if (tid < T * k) {
    const int e = __ldcg(ids + tid);   // (other CTAs may have written them)
    int rank = 0;
    for (int i = 0; i < tid; ++i) rank += __ldcg(ids + i) == e;
    const int pp = excl[e] + rank;
    pos[tid] = pp;
    src[pp] = tid;
    srow[pp] = tid / k;
  }
  __syncthreads();
  if (x_perm) {
    const int nvec = H / 8;
    for (int i = tid; i < T * k * nvec; i += NT) {
      const int r = i / nvec, v = i % nvec;
      reinterpret_cast<uint4*>(x_perm + (size_t)r * H)[v] =
          __ldg(reinterpret_cast<const uint4*>(x + (size_t)srow[r] * H) + v);
    }
  }
}

template <int NT>
static __device__ void route_tail_block(const GateParams& p, int32_t* __restrict__ counts,
                                        int32_t* __restrict__ offsets, int32_t* __restrict__ pos,
                                        int32_t* __restrict__ src, int32_t* __restrict__ active,
                                        int32_t* __restrict__ n_active,
                                        int32_t* __restrict__ shared_meta,
                                        uint16_t* __restrict__ x_perm, TailSmem& sm) {
  static_assert(NT >= kMaxExperts, "the scan takes one thread per expert");
  float* lg = sm.lg;
  int* hist = sm.hist;
  const int tid = threadIdx.x, T = p.T, C = p.C, E = p.E, k = p.k;
  const int S = p.S, n = T * C;
  const size_t stride = (size_t)T * C;

  // ---- logits: G lanes per logit (G a power of two <= 32)
  int G = 32;
  while (G > 1 && n * G > NT) G >>= 1;
  const int per = NT / G, g = tid % G;
  for (int li = tid / G; li < ((n + per - 1) / per) * per; li += per) {
    float a0 = 0.f, a1 = 0.f;
    if (li < n) {
      int sp = g;
      for (; sp + G < S; sp += 2 * G) {
        a0 += __ldcg(p.part + (size_t)sp * stride + li);
        a1 += __ldcg(p.part + (size_t)(sp + G) * stride + li);
      }
      if (sp < S) a0 += __ldcg(p.part + (size_t)sp * stride + li);
    }
    float v = a0 + a1;
    for (int o = G >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (g == 0 && li < n) lg[li] = v;
  }
  for (int e = tid; e < kMaxExperts; e += NT) hist[e] = 0;
  __syncthreads();

  // ---- gating: warp w < G_WARPS takes tokens w, w + G_WARPS, ...
  const int warp = tid >> 5;
  if (warp < G_WARPS) {
    GateParams q = p;
    q.hist = hist;
    for (int t = warp; t < T; t += G_WARPS)
      gate_token(q, t, lg + (size_t)t * C, sm.lrow[warp], sm.exact_s[warp]);
  }
  __syncthreads();

  route_dispatch_block<NT>(p.ids, T, k, E, counts, offsets, pos, src, active, n_active,
                           shared_meta, x_perm, p.x, p.H, sm);
}

}  // namespace moe

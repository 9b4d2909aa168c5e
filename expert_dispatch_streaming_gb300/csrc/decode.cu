// Fused small-batch (decode) layer forward: the whole MoE layer for T <= 16 tokens with every
// bundle resident, in one cooperative launch.
//
// At decode batch sizes a layer moves a few hundred MB of expert weights and does almost no
// arithmetic per byte, so the bound is HBM bandwidth ("The Billion-Token Bottleneck", "The
// Engineering Challenge": MoE trades compute-bound problems for IO-bound ones) -- and, with
// six dependent launches per layer, the latency of each launch boundary ("NovaLLM: Running
// Massive MoE Models Fully In-Memory", "Optimization #2": memory bandwidth and kernel launch
// overhead).  Here one persistent grid does everything and the steps meet at counters in
// global memory instead of at kernel boundaries:
//
//   router    CTA b < S bulk-copies one H slice of W_r (and of x and the shared-gate column)
//             and sums the router product over it for all tokens (fp32 partials); the last T
//             CTAs then each sum one token's partials and gate it (top-k over eight warps,
//             the exact re-scoring near the boundary as in the routing kernels); the last
//             token to be gated builds the histogram, scan, stable ranks and a route table
//             and raises a flag;
//   experts   units of one 128-row weight tile and a range of K, handed out by a grid-wide
//             counter in the order shared gate/up (needs no routing, so it streams while
//             routing runs), routed gate/up (after the flag), shared and routed down (each
//             after the gate/up tiles of its K range).  A producer warp streams the unit's
//             weight tiles with bulk asynchronous copies into a six-slot 217 KB shared-memory
//             ring (full / empty mbarriers per slot); eight consumer warps each multiply 16 of
//             the tile's rows on mma.m16n8k16 (weights as the M side, tokens on the narrow N
//             side, INT4 / NVFP4 dequantised in registers).  A unit's K range may be split:
//             the last split to arrive sums the partials in split order;
//   combine   per token, 256 columns per warp, once every down tile of the block has landed:
//             the gate-weighted sum, the shared term and the residual, and the block's sum of
//             squares; the optional RMS-normalised output once every block of the token is in.
//
// Every sum runs in a fixed order, so results do not depend on scheduling.  A warp waits only
// for units of earlier steps, every CTA is resident (cooperative launch), and every wait is
// bounded by the wall clock (~2 s): on timeout the kernel records error 9 in the workspace
// error word, every later wait gives up at once, and the producer waits (bounded) for the
// copies it issued before the CTA leaves.
#include "decode.cuh"
#include "gate.cuh"

#include <cmath>
#include <type_traits>

namespace moe {
namespace {

constexpr int kConsumerWarps = 8;                    // 8 x 16 = the 128 rows of a weight tile
constexpr int kDecThreads = 32 * (kConsumerWarps + 1);   // + one producer warp
constexpr int kColBlock = 256;                       // columns of a combine / norm unit
constexpr unsigned long long kWaitNs = 2000000000ull;
constexpr int32_t kErrDecodeWait = 9;
constexpr int kSlots = 6;                            // ring slots per CTA
constexpr int kBOff = 32768;                         // token rows after the weight tiles
constexpr int kBRowMax = 256 + 16;                   // bytes of one token row's k range (+pad)
constexpr int kSlotBytes = kBOff + kDecodeMaxT * kBRowMax;
constexpr int kSmemBytes = kSlots * kSlotBytes;      // the ring
// In a routing CTA the last kResSlots slots first hold the router slice (weights, x, shared
// gate column) and then the gating scratch; the producer fills them only once routing in the
// CTA is over.
constexpr int kResSlots = 2;
constexpr int kResOff = (kSlots - kResSlots) * kSlotBytes;
constexpr int kResBytes = kResSlots * kSlotBytes;
static_assert(sizeof(CtaGateSmem) <= (size_t)kResBytes, "gating scratch fits in the reserved slots");
static_assert(kResOff % 16 == 0, "the reserved region is 16-byte aligned");
constexpr int kRouteEntry = 8;                       // route table words per expert slot
constexpr unsigned kBackoffMaxNs = 256;              // polling back-off cap
constexpr int kGroupsMax = 32;                       // slice groups of the logit sums
constexpr int kQueue = 4;                            // unit descriptors in flight per CTA

// control words: every counter that warps poll sits on its own 128-byte line (kLine words)
constexpr int kLine = 32;
enum : int {
  kCtlRouterArrive = 0,
  kCtlGateArrive = kLine,
  kCtlRouteDone = 2 * kLine,
  kCtlNextUnit = 3 * kLine,   // the work queue: next unit to hand out
  kCtlHead = 4 * kLine   // then the route table: per expert slot {e, r0, rows, 0, 16 token bytes}
};

struct DecParams {
  GateParams g;
  const uint16_t* x;
  const uint16_t* w_gate;       // router column E: the shared-expert gate vector, or NULL
  const uint16_t* residual;
  uint16_t* out;
  uint16_t* out_n;
  float eps;
  int32_t *counts, *offsets, *pos, *src, *active, *n_active;
  BundleTable tab;
  const char* shared;
  int T, H, k, I, Is, shared_sigmoid;
  long long gu_off, dn_off, gs_off, gu_off_s, dn_off_s, gs_off_s;   // bundle byte offsets
  uint16_t *h, *y, *hs, *ys;
  float *rpart, *gpart, *dpart, *ss;   // rpart: router partials [S][T][C] (= g.part)
  int32_t *ctl, *err;
  int S, hps, Cp, Umax, Sg, Sd, Sgs, Sds, NB, mtg;    // Cp: C rounded up to 4; mtg: gate/up
                                                      // row tiles per slot
  int o_rt, o_tdone, o_gusplit, o_dnsplit, o_dnblk, o_combt;
};

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int32_t* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long wall_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool any_error(const int32_t* err) {
  return *reinterpret_cast<const volatile int32_t*>(err) != 0;
}

// The warp waits until *ctr >= target (lane 0 polls, backing off: many warps may poll one
// line).  False when this or another wait of the launch gave up: the caller skips its unit.
__device__ bool warp_wait_geq(const int32_t* ctr, int target, int32_t* err) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) {
    const unsigned long long t0 = wall_ns();
    unsigned ns = 32;
    while (ld_acquire(ctr) < target) {
      if (any_error(err)) {
        ok = 0;
        break;
      }
      if (wall_ns() - t0 > kWaitNs) {
        atomicExch(err, kErrDecodeWait);
        ok = 0;
        break;
      }
      __nanosleep(ns);
      ns = ns < kBackoffMaxNs ? 2 * ns : kBackoffMaxNs;
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);   // (lane 0's acquire + the warp barrier order the
  __syncwarp();                          //  other lanes' later loads)
  return ok != 0;
}
// Barrier of the eight consumer warps only (named barrier 1; the producer warp never joins),
// returning the AND / OR of `v` over them.
__device__ __forceinline__ int cons_and(int v) {
  int r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, 1, %2, p;\n"
      "selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(v), "n"(kConsumerWarps * 32)
      : "memory");
  return r;
}
__device__ __forceinline__ int cons_or(int v) {
  int r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.or.pred q, 1, %2, p;\n"
      "selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(v), "n"(kConsumerWarps * 32)
      : "memory");
  return r;
}
__device__ __forceinline__ void cons_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}
// Consumer thread 0 polls until *ctr >= target; the result reaches every consumer thread.
__device__ bool cons_wait_geq(const int32_t* ctr, int target, int32_t* err) {
  int ok = 1;
  if (threadIdx.x == 0) {
    const unsigned long long t0 = wall_ns();
    unsigned ns = 32;
    while (ld_acquire(ctr) < target) {
      if (any_error(err)) {
        ok = 0;
        break;
      }
      if (wall_ns() - t0 > kWaitNs) {
        atomicExch(err, kErrDecodeWait);
        ok = 0;
        break;
      }
      __nanosleep(ns);
      ns = ns < kBackoffMaxNs ? 2 * ns : kBackoffMaxNs;
    }
  }
  ok = cons_and(ok);   // (thread 0's acquire + the barrier order the other threads' loads)
  return ok != 0;
}
// The routing flag holds the number of experts with rows + 1 once routing is over.  The warp
// waits for it and gets that number, or -1 when a wait gave up.
__device__ int warp_wait_route(const int32_t* flag, int32_t* err) {
  return warp_wait_geq(flag, 1, err) ? __ldcg(flag) - 1 : -1;
}
// The warp waits until flags f[0 .. n) are all set (each lane polls its share).
__device__ bool warp_wait_flags(const int32_t* f, int n, int32_t* err) {
  const int lane = threadIdx.x & 31;
  const unsigned long long t0 = wall_ns();
  unsigned ns = 32;
  for (;;) {
    bool mine = true;
    for (int i = lane; i < n; i += 32) mine = mine && ld_acquire(f + i) >= 1;
    if (__all_sync(0xffffffffu, mine)) break;
    int stop = 0;
    if (lane == 0) {
      if (any_error(err)) {
        stop = 1;
      } else if (wall_ns() - t0 > kWaitNs) {
        atomicExch(err, kErrDecodeWait);
        stop = 1;
      }
    }
    if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    __nanosleep(ns);
    ns = ns < kBackoffMaxNs ? 2 * ns : kBackoffMaxNs;
  }
  __syncwarp();
  return true;
}
// Counter updates with release (acq_rel) semantics at GPU scope.  Issued by one thread after a
// barrier of the threads whose writes they publish: the release is cumulative over the writes
// ordered before it by the barrier.
__device__ __forceinline__ void red_release_add(int32_t* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int atom_acq_rel_add(int32_t* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}
// Publishes the warp's writes, then counts one arrival.
__device__ __forceinline__ void warp_signal(int32_t* ctr) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) red_release_add(ctr, 1);
}
// ---------------------------------------------------------------------------- mbarrier / copies
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// The same with an L2 cache policy (weights: evict first, so that the stream of expert weights
// does not push the layer's activations, counters and the kernel's own code out of L2).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Bounded wait of the whole warp for an mbarrier phase (false: timed out).  After a few quick
// tries the warp sleeps between tries, so that a waiting warp does not take issue slots from
// the warps of its SM sub-partition that have work.
__device__ __forceinline__ bool stage_wait(uint32_t bar, uint32_t parity, int32_t* err) {
  if (__all_sync(0xffffffffu, mbar_try(bar, parity))) return true;
  const unsigned long long t0 = wall_ns();
  unsigned ns = 16;
  for (uint32_t i = 1;; ++i) {
    if (__all_sync(0xffffffffu, mbar_try(bar, parity))) return true;
    if (i >= 4) {
      __nanosleep(ns);
      ns = ns < 128 ? 2 * ns : 128;
    }
    if ((i & 15) == 0) {
      const bool late = wall_ns() - t0 > kWaitNs;
      if (__any_sync(0xffffffffu, late)) {
        if ((threadIdx.x & 31) == 0) atomicExch(err, kErrDecodeWait);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

// ---------------------------------------------------------------------------- CTA ring
// Per (weight type, fused) a unit's K range is cut into blocks of KW k (one 64-k bf16 tile, one
// 128-k quantised tile), and one ring slot holds BPS blocks of every row group (gate, up) --
//   bf16 fused: 1 block x 2 tiles of 16 KB; bf16 down: 2 blocks x 1 tile;
//   quantised fused: 1 block x 2 tiles of 8448 / 9216 B; quantised down: 1 block x 1 tile --
// and, from kBOff, the same k range of the unit's token rows (rows BROW bytes apart), so the
// consumers read both operands from shared memory.
template <int WT, bool FUSED>
struct Fmt {
  static constexpr int NG = FUSED ? 2 : 1;
  static constexpr int KW = WT == 0 ? 64 : 128;
  static constexpr int TILE = WT == 0 ? 16384 : WT == 1 ? 8448 : 9216;
  static constexpr int BPS = WT == 0 ? 2 / NG : 1;
  static constexpr int BROW = BPS * KW * 2 + 16;   // +16: rows start in different banks
  static_assert(BPS * NG * TILE <= kBOff, "the tiles fit before the token rows");
  static_assert(BROW <= kBRowMax, "a token row fits its place");
};

// The unit a CTA runs: shared or routed expert (slot), 128-row tile mt, K blocks [kb_lo, kb_hi).
struct UnitRef {
  int type;        // 0 gate/up, 1 down, 2 combine, 3 normalisation, -1 nothing to do
  bool sh;         // shared expert
  int slot, mt, sp, S, kb_lo, kb_hi, t;
  const char* wsec;   // weight section of the unit's expert
  int e, r0, ne;
  int4 tok;           // the token of each of the unit's rows (bytes, row order)
};

// ---------------------------------------------------------------------------- the kernel
template <int WT, int NT>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_layer_kernel(const __grid_constant__ DecParams p) {
  extern __shared__ __align__(1024) uint8_t dsm[];
  __shared__ __align__(8) uint64_t full[kSlots], empty[kSlots], rcopy, rfree;
  __shared__ __align__(8) uint64_t qfull[kQueue], qempty[kQueue];
  __shared__ int qdesc[kQueue][2];   // unit, experts with rows (or -1: not known yet)
  __shared__ int s_flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = p.T, H = p.H, C = p.g.C, E = p.g.E, k = p.k, I = p.I, Is = p.Is;
  int32_t* ctl = p.ctl;
  // roles: CTAs [0, S) each take one H slice of the router product; the last T CTAs gate one
  // token each (gating CTA t = blockIdx.x - (gridDim.x - T)); both use the reserved slots first
  const bool routing = (int)blockIdx.x < p.S;
  const bool gating = (int)blockIdx.x >= (int)gridDim.x - T;
  const int h_lo = blockIdx.x * p.hps, h_rows = routing ? min(H, h_lo + p.hps) - h_lo : 0;
  // the router slice in the reserved slots: W_r rows [h_lo, h_lo + h_rows) (fp32, E per row),
  // then x[t][h_lo ..] for every token and the shared-expert gate column (bf16)
  uint8_t* res = dsm + kResOff;
  const float* rw = reinterpret_cast<const float*>(res);
  const uint16_t* rx = reinterpret_cast<const uint16_t*>(res + (size_t)p.hps * E * 4);
  const uint16_t* rg = rx + (size_t)T * p.hps;
  CtaGateSmem& cg = *reinterpret_cast<CtaGateSmem*>(res);   // gating, after the router step
  TailSmem& sm = cg.tail;
  const bool producer = warp == kConsumerWarps;

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kConsumerWarps);
    }
    mbar_init(smem_u32(&rcopy), 1);
    mbar_init(smem_u32(&rfree), 1);
    for (int i = 0; i < kQueue; ++i) {
      mbar_init(smem_u32(&qfull[i]), 1);
      mbar_init(smem_u32(&qempty[i]), kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  fence_proxy_async();
  __syncthreads();   // the last CTA-wide barrier: from here on the producer warp runs apart

  if (producer && routing) {
    // the router slice first, ahead of any weight tile, so that routing is not queued behind
    // the weight stream
    const uint32_t wbytes = (uint32_t)h_rows * E * 4, xbytes = (uint32_t)h_rows * 2;
    const uint32_t bar = smem_u32(&rcopy), rb = smem_u32(res);
    if (lane == 0)
      mbar_expect_tx(bar, wbytes + (uint32_t)T * xbytes + (p.w_gate ? xbytes : 0u));
    __syncwarp();
    constexpr uint32_t kChunk = 16384;
    const char* wsrc = reinterpret_cast<const char*>(p.g.w_r + (size_t)h_lo * E);
    for (uint32_t o = lane * kChunk; o < wbytes; o += 32 * kChunk)
      bulk_g2s(rb + o, wsrc + o, min(kChunk, wbytes - o), bar);
    if (lane < T)
      bulk_g2s(rb + p.hps * E * 4 + lane * p.hps * 2, p.x + (size_t)lane * H + h_lo, xbytes, bar);
    if (lane == 31 && p.w_gate)
      bulk_g2s(rb + p.hps * E * 4 + T * p.hps * 2, p.w_gate + h_lo, xbytes, bar);
  }

  if (!producer && (routing || gating)) {
    // ---------------------------------------------- router product over this CTA's H slice
    float lbv = 0.f, sbv = 0.f;   // token gating: the biases, loaded ahead
    if (gating && tid < E) {
      if (p.g.logit_bias) lbv = __ldg(p.g.logit_bias + tid);
      if (p.g.sel_bias) sbv = __ldg(p.g.sel_bias + tid);
    }
    bool ok = !routing || stage_wait(smem_u32(&rcopy), 0, p.err);
    if (routing && ok) {
      for (int c = tid; c < C; c += kConsumerWarps * 32) {
        float acc[kDecodeMaxT];
#pragma unroll
        for (int t = 0; t < kDecodeMaxT; ++t) acc[t] = 0.f;
        for (int h = 0; h < h_rows; ++h) {
          const float wv = c < E ? rw[h * E + c] : bf16_bits_to_float(rg[h]);
#pragma unroll
          for (int t = 0; t < kDecodeMaxT; ++t)
            if (t < T) acc[t] = fmaf(bf16_bits_to_float(rx[t * p.hps + h]), wv, acc[t]);
        }
#pragma unroll
        for (int t = 0; t < kDecodeMaxT; ++t)
          if (t < T) p.rpart[((size_t)blockIdx.x * T + t) * p.Cp + c] = acc[t];
      }
    }
    cons_sync();   // the router slice is read
    if (tid == 0 && routing && ok) red_release_add(ctl + kCtlRouterArrive, 1);
    // ---------------------------------------------- gating of token t
    // Two passes over the same code: pass 0, at the start of the launch while the router runs
    // elsewhere, sums whatever the partials hold and gates made-up logits (distinct, far from
    // any tie) into scratch, so that the instructions of the logit sums, the gating and the
    // dispatch are cached on this SM when pass 1 runs on the real partials.  (Run once per
    // launch, that code is otherwise fetched cold, line by line, while the weight stream loads
    // the memory system.)
    int* scr = reinterpret_cast<int*>(sm.exact_s) + 1024;   // pass-0 outputs (8 KB)
#pragma unroll 1
    for (int pass = gating ? 0 : 2; pass < 2; ++pass) {
      const bool real = pass == 1;
      const int t = real ? (int)blockIdx.x - ((int)gridDim.x - T) : 0, Tn = real ? T : 1;
      if (real && !cons_wait_geq(ctl + kCtlRouterArrive, p.S, p.err)) break;
      {
        // token t's logits: the S slice partials of four columns at a time, slice group g of
        // a quad summed by one thread in slice order (eight loads in flight), then the G
        // groups in order
        const int Cp = p.Cp, Q = Cp / 4, G = min(kGroupsMax, (kConsumerWarps * 32) / Q);
        float4* gsum = reinterpret_cast<float4*>(sm.exact_s);   // [G][Q]
        if (tid < G * Q) {
          const int q = tid % Q, g = tid / Q;
          const float4* src = reinterpret_cast<const float4*>(p.rpart + (size_t)t * Cp) + q;
          const size_t stride = (size_t)T * Cp / 4;
          float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
          int sp = g;
          for (; sp + 7 * G < p.S; sp += 8 * G) {
            float4 v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = __ldcg(src + (size_t)(sp + i * G) * stride);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              a.x += v[i].x; a.y += v[i].y; a.z += v[i].z; a.w += v[i].w;
            }
          }
          for (; sp < p.S; sp += G) {
            const float4 v = __ldcg(src + (size_t)sp * stride);
            a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
          }
          gsum[g * Q + q] = a;
        }
        cons_sync();
        if (tid < Q) {
          float4 a = gsum[tid];
          for (int g = 1; g < G; ++g) {
            const float4 v = gsum[g * Q + tid];
            a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
          }
          reinterpret_cast<float4*>(sm.lg)[tid] = a;
        }
      }
      if (!real) {
        cons_sync();
        for (int c = tid; c < C; c += kConsumerWarps * 32) sm.lg[c] = -0.5f * (float)c;
      }
      for (int e = tid; e < kMaxExperts; e += kConsumerWarps * 32) {
        sm.hist[e] = 0;
        cg.gc.lb[e] = real ? lbv : 0.f;
        cg.gc.sb[e] = real ? sbv : 0.f;
      }
      cons_sync();
      GateParams q = p.g;
      q.hist = sm.hist;
      int* ids_s = sm.srow;                         // Tn * k ids
      if (Tn == 1) q.ids_local = ids_s;
      // where this pass writes: the real outputs, or scratch
      int32_t* o_counts = real ? p.counts : scr + 16;
      int32_t* o_offsets = real ? p.offsets : scr + 272;
      int32_t* o_active = real ? p.active : scr + 529;
      int32_t* o_pos = real ? p.pos : scr + 785;
      int32_t* o_src = real ? p.src : scr + 913;
      int32_t* o_nact = real ? p.n_active : scr + 1041;
      int32_t* o_rt = real ? ctl + p.o_rt : scr + 1042;
      if (!real) {
        q.ids = scr;
        q.w = reinterpret_cast<float*>(scr + 8);
        q.forced = nullptr;
        q.logits = nullptr;
        q.shared_gate = nullptr;
        q.tie_flags = nullptr;
      }
      gate_token_cta<kConsumerWarps * 32>(q, t, sm.lg, cg.gc, sm.lrow[0], sm.exact_s[0],
                                          [] { cons_sync(); });
      if (tid == 0) s_flag = Tn == 1 || atom_acq_rel_add(ctl + kCtlGateArrive, 1) == T - 1;
      cons_sync();
      if (s_flag) {
        // the last token gated: every id is visible.  Histogram, scan, ranks, route table.
        int* rt = reinterpret_cast<int*>(sm.lrow);    // route table being built
        if (Tn > 1)
          for (int i = tid; i < Tn * k; i += kConsumerWarps * 32) ids_s[i] = __ldcg(p.g.ids + i);
        for (int e = tid; e < kMaxExperts; e += kConsumerWarps * 32) sm.hist[e] = 0;
        cons_sync();
        for (int i = tid; i < Tn * k; i += kConsumerWarps * 32) atomicAdd(&sm.hist[ids_s[i]], 1);
        cons_sync();
        // one pass of scans over the experts: rows (low 16 bits) and experts with rows
        static_assert(kConsumerWarps * 32 >= kMaxExperts, "one thread per expert");
        const int cnt = tid < E ? sm.hist[tid] : 0;
        int v = cnt + (cnt > 0 ? 0x10000 : 0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, v, o);
          if (lane >= o) v += y;
        }
        if (lane == 31) sm.excl[warp] = v;
        cons_sync();
        int base = 0;
        for (int w = 0; w < warp; ++w) base += sm.excl[w];
        v += base;                                   // inclusive
        const int off = (v & 0xffff) - cnt, slot = (v >> 16) - 1;
        cons_sync();
        if (tid < E) {
          sm.excl[tid] = off;
          o_counts[tid] = cnt;
          o_offsets[tid] = off;
          if (tid == E - 1) {
            o_offsets[E] = off + cnt;
            *o_nact = slot + 1;
            s_flag = slot + 1;
          }
          if (cnt > 0) {
            o_active[slot] = tid;
            int* en = rt + slot * kRouteEntry;
            en[0] = tid;
            en[1] = off;
            en[2] = cnt;
            en[3] = en[4] = en[5] = en[6] = en[7] = 0;
            cg.gc.rank[tid] = slot;                     // expert -> slot
          }
        }
        cons_sync();
        // stable ranks: pair i goes after every earlier pair routed to its expert
        for (int i = tid; i < Tn * k; i += kConsumerWarps * 32) {
          const int e = ids_s[i];
          int rank = 0;
          for (int j = 0; j < i; ++j) rank += ids_s[j] == e;
          const int pp = sm.excl[e] + rank;
          o_pos[i] = pp;
          o_src[pp] = i;
          if (rank < kDecodeMaxT)   // (forced ids may repeat an expert within a token)
            reinterpret_cast<uint8_t*>(rt + cg.gc.rank[e] * kRouteEntry + 4)[rank] = (uint8_t)(i / k);
        }
        cons_sync();
        const int n_act = s_flag;
        for (int w = tid; w < n_act * kRouteEntry; w += kConsumerWarps * 32) o_rt[w] = rt[w];
        cons_sync();
        if (tid == 0 && real) st_release(ctl + kCtlRouteDone, n_act + 1);
      }
      cons_sync();
    }
    cons_sync();
    if (tid == 0) mbar_arrive(smem_u32(&rfree));   // the reserved slots go to the ring
  }

  const int MTg = I / 128, MTs = Is / 128, MTd = H / 128;
  const int nA = Is ? MTs * p.Sgs : 0;   // shared gate/up
  const int nC = Is ? MTd * p.Sds : 0;   // shared down
  const int nB = p.Umax * MTg * p.Sg;    // routed gate/up
  const int nD = p.Umax * MTd * p.Sd;    // routed down
  const int nE = T;
  const int nF = p.out_n ? T : 0;
  const int total = nA + nC + nB + nD + nE + nF;
  const int shared_slot = p.Umax;
  const int32_t* rtab = ctl + p.o_rt;
  int32_t* tdone = ctl + p.o_tdone;
  int32_t* gu_split = ctl + p.o_gusplit;
  int32_t* dn_split = ctl + p.o_dnsplit;
  int32_t* dn_blk = ctl + p.o_dnblk;
  int32_t* comb_t = ctl + p.o_combt;

  // The unit u of the schedule, in the order shared gate/up, routed gate/up, shared down,
  // routed down, combine, normalisation (the same decoding in the producer and the consumers):
  // the shared expert's gate/up needs no routing, so it streams while routing runs, and every
  // gate/up unit is handed out before the down units that wait for it.  Routed
  // units resolve their expert from the route table (n_act >= 0: routing is over, n_act experts
  // have rows); a routed slot beyond them has nothing to do.
  auto unit_of = [&](int u, int n_act) -> UnitRef {
    UnitRef r{};
    r.type = -1;
    int v = u;
    bool down;
    if (v < nA) {
      r.sh = true;
      down = false;
    } else if (v < nA + nB) {
      r.sh = false;
      down = false;
      v -= nA;
    } else if (v < nA + nB + nC) {
      r.sh = true;
      down = true;
      v -= nA + nB;
    } else if (v < nA + nB + nC + nD) {
      r.sh = false;
      down = true;
      v -= nA + nB + nC;
    } else if (v < nA + nC + nB + nD + nE) {
      r.type = 2;
      r.t = v - (nA + nC + nB + nD);
      return r;
    } else {
      r.type = 3;
      r.t = v - (nA + nC + nB + nD + nE);
      return r;
    }
    r.type = down ? 1 : 0;
    r.S = down ? (r.sh ? p.Sds : p.Sd) : (r.sh ? p.Sgs : p.Sg);
    r.sp = v % r.S;
    v /= r.S;
    const int MT = down ? MTd : (r.sh ? MTs : MTg);
    r.mt = v % MT;
    r.slot = r.sh ? shared_slot : v / MT;
    const int KW = down ? Fmt<WT, false>::KW : Fmt<WT, true>::KW;
    const int KB = (down ? (r.sh ? Is : I) : H) / KW, per = (KB + r.S - 1) / r.S;
    r.kb_lo = r.sp * per;
    r.kb_hi = min(KB, r.kb_lo + per);
    if (r.sh) {
      r.e = -1;
      r.r0 = 0;
      r.ne = T;
      r.tok = make_int4(0x03020100, 0x07060504, 0x0b0a0908, 0x0f0e0d0c);
      r.wsec = p.shared + (down ? p.dn_off_s : p.gu_off_s);
      return r;
    }
    if (n_act < 0) return r;
    if (n_act <= r.slot) {
      r.type = -1;
      return r;
    }
    const int4 a = __ldcg(reinterpret_cast<const int4*>(rtab + r.slot * kRouteEntry));
    r.tok = __ldcg(reinterpret_cast<const int4*>(rtab + r.slot * kRouteEntry + 4));
    r.e = a.x;
    r.r0 = a.y;
    r.ne = min(a.z, 8 * NT);   // <= T: one row per token
    r.wsec = static_cast<const char*>(p.tab.p[r.e]) + (down ? p.dn_off : p.gu_off);
    return r;
  };

  if (producer) {
    // ---------------------------------------------- producer: bulk copies of weight tiles
    // Units come from one work queue for the whole grid (a counter in global memory), in the
    // order of the schedule; each is announced to the consumers through a shared-memory
    // descriptor queue before its tiles are issued.  A CTA that gates a token takes its first
    // unit only once gating is over, so no unit that others wait for sits behind it.
    uint32_t used = 0, epar = 0, qused = 0, qpar = 0;
    int gs = 0, qi = 0;   // stages issued, descriptors pushed
    const uint64_t wpol = policy_evict_first();
    bool ok = true, res_free = !(routing || gating);
    int n_act = -1;
    auto push = [&](int u, int na) -> bool {
      const int i = qi % kQueue;
      if ((qused >> i) & 1u) {
        if (!stage_wait(smem_u32(&qempty[i]), (qpar >> i) & 1u, p.err)) return false;
        qpar ^= 1u << i;
      }
      qused |= 1u << i;
      if (lane == 0) {
        qdesc[i][0] = u;
        qdesc[i][1] = na;
        mbar_arrive(smem_u32(&qfull[i]));
      }
      __syncwarp();
      ++qi;
      return true;
    };
    auto grab = [&]() -> int {
      int v = 0;
      if (lane == 0) v = atomicAdd(ctl + kCtlNextUnit, 1);
      return __shfl_sync(0xffffffffu, v, 0);
    };
    if (gating) {
      ok = stage_wait(smem_u32(&rfree), 0, p.err);
      res_free = true;
    }
    int u = ok ? grab() : total;
    while (ok && u < total) {
      const int u_next = grab();   // (its latency overlaps this unit's issue)
      UnitRef r = unit_of(u, -1);
      if ((r.type <= 1 && !r.sh) || r.type == 2) {
        if (n_act < 0 && (n_act = warp_wait_route(ctl + kCtlRouteDone, p.err)) < 0) break;
        r = unit_of(u, n_act);
      }
      if (r.type < 0 || r.type > 1) {
        if (r.type >= 0 && !push(u, n_act)) break;
        u = u_next;
        continue;
      }
      const bool fused = r.type == 0;
      const int BPS = fused ? Fmt<WT, true>::BPS : Fmt<WT, false>::BPS;
      const int BROW = fused ? Fmt<WT, true>::BROW : Fmt<WT, false>::BROW;
      const int NG = fused ? 2 : 1;
      constexpr int TILE = Fmt<WT, true>::TILE;
      constexpr int KW = Fmt<WT, true>::KW;
      const int K = fused ? H : (r.sh ? Is : I);
      const int KT = K / KW;                                 // tiles along K per row tile
      const int Mup = (r.sh ? Is : I) / 128;                 // up rows' first row tile
      // this lane's token row (the unit's rows are its tokens' x rows, or its h rows)
      const uint16_t* brow = nullptr;
      if (lane < r.ne) {
        const int tw = lane < 8 ? (lane < 4 ? r.tok.x : r.tok.y) : (lane < 12 ? r.tok.z : r.tok.w);
        const int tok = (tw >> (8 * (lane & 3))) & 0xff;
        if (fused) brow = p.x + (size_t)tok * H;
        else brow = r.sh ? p.hs + (size_t)lane * Is : p.h + (size_t)(r.r0 + lane) * I;
      }
      // a down unit's K range of h comes from other CTAs' gate/up tiles; its first weight
      // tiles are already on their way when the producer waits for those
      bool h_ready = fused;
      const int t_lo = r.kb_lo * KW / 128, t_hi = (r.kb_hi * KW + 127) / 128;
      if (!push(u, n_act)) break;
      for (int kb = r.kb_lo; kb < r.kb_hi; kb += BPS) {
        const int s = gs % kSlots;
        if (!res_free && s >= kSlots - kResSlots) {
          // the reserved slots: only once routing in this CTA is over
          if (!stage_wait(smem_u32(&rfree), 0, p.err)) {
            ok = false;
            break;
          }
          res_free = true;
        }
        if ((used >> s) & 1u) {
          if (!stage_wait(smem_u32(&empty[s]), (epar >> s) & 1u, p.err)) {
            ok = false;
            break;
          }
          epar ^= 1u << s;
        }
        used |= 1u << s;
        const int nkb = min(BPS, r.kb_hi - kb);
        const uint32_t bar = smem_u32(&full[s]), sb = smem_u32(dsm) + s * kSlotBytes;
        const uint32_t brow_bytes = (uint32_t)nkb * KW * 2;
        if (lane == 0) mbar_expect_tx(bar, (uint32_t)(nkb * NG * TILE) + r.ne * brow_bytes);
        __syncwarp();
        if (lane < nkb * NG) {
          const int b = lane / NG, q = lane % NG;
          const int rt = r.mt + (q ? Mup : 0);
          const char* src = r.wsec + ((size_t)rt * KT + kb + b) * TILE;
          bulk_g2s_hint(sb + (b * NG + q) * TILE, src, TILE, bar, wpol);
        }
        if (!h_ready) {
          // wait for the gate/up tiles, then order their generic-proxy writes of h before
          // this warp's bulk (async-proxy) reads of it
          if (!warp_wait_flags(tdone + r.slot * p.mtg + t_lo, t_hi - t_lo, p.err)) {
            ok = false;
            break;
          }
          asm volatile("fence.proxy.async.global;" ::: "memory");
          h_ready = true;
        }
        if (brow != nullptr) bulk_g2s(sb + kBOff + lane * BROW, brow + (size_t)kb * KW, brow_bytes, bar);
        ++gs;
      }
      u = u_next;
    }
    push(-1, 0);   // the end of this CTA's units
    // no copy may land after the CTA is gone: wait (bounded) for the router slice and the
    // last fill of each slot
    const unsigned long long t0 = wall_ns();
    if (routing)
      while (!__all_sync(0xffffffffu, mbar_try(smem_u32(&rcopy), 0)))
        if (wall_ns() - t0 > kWaitNs) break;
    for (int s = 0; s < kSlots; ++s) {
      const int n = gs / kSlots + (s < gs % kSlots ? 1 : 0);   // fills of slot s
      if (n == 0) continue;
      while (!__all_sync(0xffffffffu, mbar_try(smem_u32(&full[s]), (uint32_t)((n - 1) & 1))))
        if (wall_ns() - t0 > kWaitNs) break;
    }
    return;
  }

  // ------------------------------------------------ consumers: 8 warps, 16 weight rows each
  const int g = lane >> 2, tq = lane & 3;
  uint32_t fpar = 0, qpar = 0;
  int cs = 0, qi = 0;   // stages consumed, descriptors taken
  for (;;) {
    // the next unit from the producer (routed ones already resolved)
    const int qs = qi % kQueue;
    if (!stage_wait(smem_u32(&qfull[qs]), (qpar >> qs) & 1u, p.err)) break;
    qpar ^= 1u << qs;
    const int u = qdesc[qs][0], n_act = qdesc[qs][1];
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&qempty[qs]));
    ++qi;
    if (u < 0) break;
    const UnitRef r = unit_of(u, n_act);
    if (r.type < 0) continue;
    if (r.type <= 1) {
      const bool fused = r.type == 0;
      // accumulators: gate (or down) and up rows, even and odd k steps apart, so that the MMAs
      // of a block form two independent chains per tile
      float acc[NT][4], accu[NT][4], acc2[NT][4], accu2[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[j][q] = accu[j][q] = acc2[j][q] = accu2[j][q] = 0.f;
      constexpr int TILE = Fmt<WT, true>::TILE;
      constexpr int KW = Fmt<WT, true>::KW;
      constexpr int XV = KW / 32;     // 16-byte pieces of a token row per lane and block
      constexpr int STEPS = KW / 16;  // k steps of 16 per block
      // One stage: NGc row groups (2: gate and up tiles, 1: down) of nkb blocks.  Plain
      // shared-memory loads and non-volatile MMAs, so that the compiler may overlap the loads
      // and dequantisation of one tile with the MMAs of the other.
      auto run_stage = [&](auto ngc, const uint8_t* sl, int nkb) {
        constexpr int NGc = decltype(ngc)::value;
        constexpr int BROWc = Fmt<WT, NGc == 2>::BROW;
        for (int b = 0; b < nkb; ++b) {
          // token fragments: the lane's KW / 4 k of the block for token rows 8 j + g
          uint4 xb[NT][XV];
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            const int n = 8 * j + g;
#pragma unroll
            for (int v = 0; v < XV; ++v) {
              // bf16: chunks 2 tq, 2 tq + 1 of the block (k = 16 tq ..); quantised: the lane's
              // word v of each 32-k chunk (k = 32 v + 8 tq ..), the k order of its weight words
              const int k0 = WT == 0 ? (KW / 4) * tq + 8 * v : 32 * v + 8 * tq;
              xb[j][v] = n < r.ne ? *reinterpret_cast<const uint4*>(
                                        sl + kBOff + n * BROWc + (b * KW + k0) * 2)
                                  : make_uint4(0, 0, 0, 0);
            }
          }
#pragma unroll
          for (int q = 0; q < NGc; ++q) {
            const uint8_t* tb = sl + (b * NGc + q) * TILE;
            // weight fragments of rows w*16 + g (+8) of this tile
            uint32_t af[STEPS][2][2];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int rr = warp * 16 + g + 8 * h2;
              if constexpr (WT == 0) {
                uint4 a4[2];
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                  const int c = 2 * tq + v;
                  a4[v] = *reinterpret_cast<const uint4*>(tb + rr * 128 + ((c ^ (rr & 7)) << 4));
                }
#pragma unroll
                for (int st = 0; st < STEPS; ++st) {
                  af[st][h2][0] = word_of(a4[st >> 1], (2 * st) & 3);
                  af[st][h2][1] = word_of(a4[st >> 1], (2 * st + 1) & 3);
                }
              } else {
                // One ldmatrix of four 8 x 16-byte matrices, matrix i = the 32-code chunks i of
                // rows rr - g .. rr - g + 7: the lane gets word tq of chunk i of its row rr for
                // i = 0..3 (codes k = 32 i + 8 tq .. + 7), with each matrix's eight rows in
                // distinct bank groups (a lane's own chunk tq of its row would put the four
                // lanes of a row on one bank group)
                uint4 a4;
                asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                             : "=r"(a4.x), "=r"(a4.y), "=r"(a4.z), "=r"(a4.w)
                             : "r"(smem_u32(tb) +
                                   (((lane >> 3) * 128 + warp * 16 + (lane & 7) + 8 * h2) << 4)));
                uint32_t scw[4];   // the scale pair of each of the lane's four words
                if constexpr (WT == 1) {
                  scw[0] = int4_scale_pair(*reinterpret_cast<const uint16_t*>(tb + 8192 + 2 * rr));
                  scw[1] = scw[2] = scw[3] = scw[0];
                } else {
                  // the row's 8 block scales (16 k each): word i's is block 2 i + tq / 2
                  const uint2 eight = *reinterpret_cast<const uint2*>(tb + 8192 + 8 * rr);
                  const int hi = tq >> 1;
                  scw[0] = fp4_scale_pair(eight.x, hi);
                  scw[1] = fp4_scale_pair(eight.x, 2 + hi);
                  scw[2] = fp4_scale_pair(eight.y, hi);
                  scw[3] = fp4_scale_pair(eight.y, 2 + hi);
                }
#pragma unroll
                for (int st = 0; st < STEPS; ++st) {
                  // step st: codes 4st .. 4st+3 of the lane's 32 = word st / 2, pairs (st & 1) * 2, + 1
                  const uint32_t wq = word_of(a4, st >> 1);
                  const uint32_t scp = scw[st >> 1];
                  if constexpr (WT == 1) {
                    af[st][h2][0] = int4_pair_dyn(wq, (st & 1) * 2, scp);
                    af[st][h2][1] = int4_pair_dyn(wq, (st & 1) * 2 + 1, scp);
                  } else if ((st & 1) == 0) {
                    af[st][h2][0] = fp4_pair<0>(wq, scp);
                    af[st][h2][1] = fp4_pair<1>(wq, scp);
                  } else {
                    af[st][h2][0] = fp4_pair<2>(wq, scp);
                    af[st][h2][1] = fp4_pair<3>(wq, scp);
                  }
                }
              }
            }
#pragma unroll
            for (int st = 0; st < STEPS; ++st)
#pragma unroll
              for (int j = 0; j < NT; ++j) {
                const uint32_t b0 = word_of(xb[j][st >> 1], (2 * st) & 3);
                const uint32_t b1 = word_of(xb[j][st >> 1], (2 * st + 1) & 3);
                float(&d)[4] = q == 0 ? ((st & 1) ? acc2[j] : acc[j]) : ((st & 1) ? accu2[j] : accu[j]);
                mma16816(d, af[st][0][0], af[st][1][0], af[st][0][1], af[st][1][1], b0, b1);
              }
          }
        }
      };
      const int BPS = fused ? Fmt<WT, true>::BPS : Fmt<WT, false>::BPS;
      bool ok = true;
      for (int kb = r.kb_lo; kb < r.kb_hi; kb += BPS) {
        const int s = cs % kSlots;
        if (!stage_wait(smem_u32(&full[s]), (fpar >> s) & 1u, p.err)) {
          ok = false;
          break;
        }
        fpar ^= 1u << s;
        const uint8_t* sl = dsm + s * kSlotBytes;
        const int nkb = min(BPS, r.kb_hi - kb);
        if (fused) run_stage(std::integral_constant<int, 2>{}, sl, nkb);
        else run_stage(std::integral_constant<int, 1>{}, sl, nkb);
        // the slot is read (the arrive releases the warp's reads of it to the producer)
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        ++cs;
      }
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[j][q] += acc2[j][q];
          accu[j][q] += accu2[j][q];
        }
      if (!ok) break;
      // ---------------------------------------------- epilogue of a 128-row tile
      const int Mo = fused ? (r.sh ? Is : I) : H;
      float fa = 1.f, fb = 1.f;   // NVFP4 matrix scales (x 2^7)
      if (WT == 2) {
        const char* bb = r.sh ? p.shared : static_cast<const char*>(p.tab.p[r.e]);
        const float* gsv = reinterpret_cast<const float*>(bb + (r.sh ? p.gs_off_s : p.gs_off));
        fa = __ldg(gsv + (fused ? 0 : 2)) * 128.f;
        fb = __ldg(gsv + 1) * 128.f;
      }
      uint16_t* outp = fused ? (r.sh ? p.hs : p.h) : (r.sh ? p.ys : p.y);
      const int ne = r.ne;
      if (r.S > 1) {
        const int smax = fused ? max(p.Sg, p.Sgs) : max(p.Sd, p.Sds);
        const int grp = r.slot * (fused ? p.mtg : MTd) + r.mt;
        const int pw = fused ? 256 : 128;   // partial row: gate then up columns (fused)
        float* base = (fused ? p.gpart : p.dpart) + (size_t)grp * smax * 16 * pw;
        float* pp = base + (size_t)r.sp * 16 * pw;
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int n = 8 * j + 2 * tq + (q & 1), m = warp * 16 + g + 8 * (q >> 1);
            if (n < ne) {
              pp[n * pw + m] = acc[j][q];
              if (fused) pp[n * pw + 128 + m] = accu[j][q];
            }
          }
        cons_sync();
        int last = 0;
        if (tid == 0) last = atom_acq_rel_add((fused ? gu_split : dn_split) + grp, 1) == r.S - 1;
        if (!cons_or(last)) continue;
        for (int i = tid; i < ne * 128; i += kConsumerWarps * 32) {
          const int n = i >> 7, m = i & 127;
          float a0 = 0.f, a1 = 0.f;
          for (int q = 0; q < r.S; ++q) {
            a0 += __ldcg(base + ((size_t)q * 16 + n) * pw + m);
            if (fused) a1 += __ldcg(base + ((size_t)q * 16 + n) * pw + 128 + m);
          }
          const float v = fused ? silu_mul(a0 * fa, a1 * fb) : a0 * fa;
          outp[(size_t)(r.r0 + n) * Mo + r.mt * 128 + m] = float_to_bf16_bits(v);
        }
      } else {
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int n = 8 * j + 2 * tq + (q & 1), m = warp * 16 + g + 8 * (q >> 1);
            if (n < ne) {
              const float v = fused ? silu_mul(acc[j][q] * fa, accu[j][q] * fb) : acc[j][q] * fa;
              outp[(size_t)(r.r0 + n) * Mo + r.mt * 128 + m] = float_to_bf16_bits(v);
            }
          }
      }
      cons_sync();
      if (tid == 0) {
        if (fused) st_release(tdone + r.slot * p.mtg + r.mt, 1);
        else red_release_add(dn_blk + (r.mt * 128) / kColBlock * kLine, 1);
      }
    } else if (r.type == 2) {
      // ---------------------------------------------- combine of token t, 256 columns per warp
      const int t = r.t;
      for (int b = warp; b < p.NB; b += kConsumerWarps) {
        const int tiles = (min(kColBlock, H - b * kColBlock) + 127) / 128;
        if (!warp_wait_geq(dn_blk + b * kLine, tiles * (n_act + (Is ? 1 : 0)), p.err)) break;
        const int c = b * kColBlock + 8 * lane;
        float ssq = 0.f;
        if (c < H) {
          float acc8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          uint4 q4[kMaxK];
          float wj[kMaxK];
#pragma unroll
          for (int j = 0; j < kMaxK; ++j) {
            q4[j] = make_uint4(0, 0, 0, 0);
            wj[j] = 0.f;
            if (j < k) {
              const int pj = __ldcg(p.pos + t * k + j);
              wj[j] = __ldcg(p.g.w + t * k + j);
              q4[j] = __ldcg(reinterpret_cast<const uint4*>(p.y + (size_t)pj * H + c));
            }
          }
#pragma unroll
          for (int j = 0; j < kMaxK; ++j) {
            if (j < k) {
              const uint32_t qw[4] = {q4[j].x, q4[j].y, q4[j].z, q4[j].w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 f = bf16x2_to_float2(qw[i]);
                acc8[2 * i] = fmaf(wj[j], f.x, acc8[2 * i]);
                acc8[2 * i + 1] = fmaf(wj[j], f.y, acc8[2 * i + 1]);
              }
            }
          }
          if (Is) {
            const float gsh = p.shared_sigmoid ? __ldcg(p.g.shared_gate + t) : 1.f;
            const uint4 s4 = __ldcg(reinterpret_cast<const uint4*>(p.ys + (size_t)t * H + c));
            const uint32_t qw[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = bf16x2_to_float2(qw[i]);
              acc8[2 * i] = fmaf(gsh, f.x, acc8[2 * i]);
              acc8[2 * i + 1] = fmaf(gsh, f.y, acc8[2 * i + 1]);
            }
          }
          uint4 rq = make_uint4(0, 0, 0, 0);
          if (p.residual) rq = __ldg(reinterpret_cast<const uint4*>(p.residual + (size_t)t * H + c));
          const uint32_t rw[4] = {rq.x, rq.y, rq.z, rq.w};
          uint32_t o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t bb = float2_to_bf16x2(acc8[2 * i], acc8[2 * i + 1]);
            if (p.residual) {
              const float2 rr = bf16x2_to_float2(rw[i]);
              const float2 f = bf16x2_to_float2(bb);
              bb = float2_to_bf16x2(rr.x + f.x, rr.y + f.y);
            }
            o[i] = bb;
            const float2 f = bf16x2_to_float2(bb);
            ssq = fmaf(f.x, f.x, fmaf(f.y, f.y, ssq));
          }
          reinterpret_cast<uint4*>(p.out + (size_t)t * H)[c / 8] = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (p.out_n) {
#pragma unroll
          for (int d = 16; d > 0; d >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, d);
          if (lane == 0) p.ss[(size_t)b * T + t] = ssq;
          warp_signal(comb_t + t * kLine);
        }
      }
    } else {
      // ---------------------------------------------- RMS normalisation of token t
      const int t = r.t;
      if (!warp_wait_geq(comb_t + t * kLine, p.NB, p.err)) break;
      float ssum = 0.f;
      for (int i = lane; i < p.NB; i += 32) ssum += __ldcg(p.ss + (size_t)i * T + t);
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, d);
      const float scale = 1.f / sqrtf(ssum / (float)H + p.eps);
      for (int b = warp; b < p.NB; b += kConsumerWarps) {
        const int c = b * kColBlock + 8 * lane;
        if (c < H) {
          const uint4 q4 = __ldcg(reinterpret_cast<const uint4*>(p.out + (size_t)t * H + c));
          const uint32_t qw[4] = {q4.x, q4.y, q4.z, q4.w};
          uint32_t o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = bf16x2_to_float2(qw[i]);
            o[i] = float2_to_bf16x2(f.x * scale, f.y * scale);
          }
          reinterpret_cast<uint4*>(p.out_n + (size_t)t * H)[c / 8] =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
  }
}

template <int WT, int NT>
int blocks_per_sm() {
  static int n = -1;
  if (n < 0) {
    int b = 0;
    if (cudaFuncSetAttribute(decode_layer_kernel<WT, NT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, decode_layer_kernel<WT, NT>,
                                                      kDecThreads, kSmemBytes) != cudaSuccess) {
      cudaGetLastError();
      b = 0;
    }
    n = b;
  }
  return n;
}

template <int WT, int NT>
cudaError_t launch_wt(const DecParams& dp, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_layer_kernel<WT, NT>, dp);
}

int bps_of(int wt, int nt) {
  if (wt == 0) return nt == 1 ? blocks_per_sm<0, 1>() : blocks_per_sm<0, 2>();
  if (wt == 1) return nt == 1 ? blocks_per_sm<1, 1>() : blocks_per_sm<1, 2>();
  return nt == 1 ? blocks_per_sm<2, 1>() : blocks_per_sm<2, 2>();
}

// K split of `units` CTA units over `G` CTAs: the launch takes ~ ceil(units * S / G) waves of
// 1/S of the K range each (the partial sums cost a little per extra split)
int best_split(int units, int KB, int G) {
  int best_s = 1;
  double best = (double)ceil_div(units, G);
  for (int s = 2; s <= std::min(KB, 32); ++s) {
    const double c = (double)ceil_div(units * s, G) / s * (1.0 + 0.03 * (s - 1));
    if (c < best * 0.97) {
      best = c;
      best_s = s;
    }
  }
  const int per = ceil_div(KB, best_s);
  return ceil_div(KB, per);
}

}  // namespace

DecodePlan plan_decode(int T, int H, int E, int k, int I, int Is, int wdtype, bool has_gate) {
  DecodePlan p{};
  p.ok = T >= 1 && T <= kDecodeMaxT && H % 128 == 0 && I % 128 == 0 && Is % 128 == 0 &&
         E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E && wdtype >= 0 &&
         wdtype <= 2;
  if (!p.ok) return p;
  const int nt = T <= 8 ? 1 : 2;
  if (bps_of(wdtype, nt) < 1) {   // one CTA (one 216 KB ring) per SM
    p.ok = 0;
    return p;
  }
  p.grid = sm_count();
  p.C = E + (has_gate ? 1 : 0);
  p.Cp = (int)round_up((size_t)p.C, 4);
  // router slices: one per CTA, each a multiple of 8 rows (16-byte bulk copies of the bf16
  // x and gate columns), and the slice (W_r rows, x and gate columns) must fit the reserved slots
  p.hps = (int)round_up((size_t)ceil_div(H, p.grid - T), 8);
  auto slice_bytes = [&](int hps) { return (size_t)hps * (E * 4 + (T + 1) * 2); };
  if (slice_bytes(p.hps) > (size_t)kResBytes) {
    p.ok = 0;
    return p;
  }
  p.S = ceil_div(H, p.hps);
  if (p.S > p.grid - T) {   // the gating CTAs take no router slice
    p.ok = 0;
    return p;
  }
  p.Umax = std::min(E, T * k);
  const int KW = wdtype == 0 ? 64 : 128;
  // the splits are chosen for the expected number of experts with rows under uniform routing,
  // E (1 - (1 - k/E)^T), not the bound Umax (the buffers are sized by Umax)
  const double p_used = 1.0 - std::pow(1.0 - (double)k / E, (double)T);
  const int U_est = std::max(1, std::min(p.Umax, (int)std::ceil(E * p_used - 1e-9)));
  const int ngu = U_est * (I / 128) + Is / 128;
  p.Sg = best_split(ngu, H / KW, p.grid);
  p.Sgs = p.Sg;
  const int ndn = (U_est + (Is ? 1 : 0)) * (H / 128);
  p.Sd = best_split(ndn, I / KW, p.grid);
  p.Sds = Is ? best_split(ndn, Is / KW, p.grid) : 1;
  p.NB = ceil_div(H, kColBlock);
  const int mtg = std::max(I, Is) / 128;
  const int slots = p.Umax + 1;
  const int sgm = std::max(p.Sg, p.Sgs), sdm = std::max(p.Sd, p.Sds);
  p.gpart_elems = sgm > 1 ? (size_t)slots * mtg * sgm * 16 * 256 : 1;
  p.dpart_elems = sdm > 1 ? (size_t)slots * (H / 128) * sdm * 16 * 128 : 1;
  p.ctl_words = kCtlHead + (size_t)p.Umax * kRouteEntry + 2 * (size_t)slots * mtg +
                (size_t)slots * (H / 128) + (size_t)p.NB * kLine + (size_t)T * kLine;
  return p;
}

int launch_decode(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t st) {
  if (!pl.ok) return MOE_ERR_UNSUPPORTED;
  DecParams p{};
  GateParams& gp = p.g;
  gp.part = a.part; gp.S = pl.S; gp.C = pl.C; gp.ldp = pl.C;
  gp.x = a.x; gp.w_r = a.w_r; gp.w_rT = nullptr; gp.logit_bias = a.logit_bias;
  gp.sel_bias = a.sel_bias; gp.forced = a.forced; gp.T = a.T; gp.H = a.H; gp.E = a.E; gp.k = a.k;
  gp.mode = a.gating; gp.scale = a.scale; gp.ids = a.ids; gp.w = a.w; gp.logits = nullptr;
  gp.shared_gate = a.shared_gate; gp.tie_flags = a.tie; gp.hist = nullptr;
  p.x = a.x; p.w_gate = a.w_gate; p.residual = a.residual; p.out = a.out; p.out_n = a.out_n;
  p.eps = a.eps;
  p.counts = a.counts; p.offsets = a.offsets; p.pos = a.pos; p.src = a.src;
  p.active = a.active; p.n_active = a.n_active;
  p.tab = a.tab;
  p.shared = static_cast<const char*>(a.shared);
  p.T = a.T; p.H = a.H; p.k = a.k; p.I = a.I; p.Is = a.Is; p.shared_sigmoid = a.shared_sigmoid;
  p.gu_off = (long long)a.lay.gate_up_offset;
  p.dn_off = (long long)a.lay.down_offset;
  p.gs_off = (long long)a.lay.global_scale_offset;
  p.gu_off_s = (long long)a.slay.gate_up_offset;
  p.dn_off_s = (long long)a.slay.down_offset;
  p.gs_off_s = (long long)a.slay.global_scale_offset;
  p.h = a.h; p.y = a.y; p.hs = a.hs; p.ys = a.ys;
  p.rpart = a.part; p.gpart = a.gpart; p.dpart = a.dpart; p.ss = a.ss;
  p.ctl = a.ctl; p.err = a.err;
  p.S = pl.S; p.hps = pl.hps; p.Cp = pl.Cp; p.Umax = pl.Umax; p.Sg = pl.Sg; p.Sd = pl.Sd; p.Sgs = pl.Sgs;
  p.Sds = pl.Sds; p.NB = pl.NB;
  p.mtg = std::max(a.I, a.Is) / 128;
  const int slots = pl.Umax + 1;
  p.o_rt = kCtlHead;
  p.o_tdone = p.o_rt + pl.Umax * kRouteEntry;
  p.o_gusplit = p.o_tdone + slots * p.mtg;
  p.o_dnsplit = p.o_gusplit + slots * p.mtg;
  p.o_dnblk = p.o_dnsplit + slots * (a.H / 128);
  p.o_combt = p.o_dnblk + pl.NB * kLine;
  const int nt = a.T <= 8 ? 1 : 2;
  cudaError_t e;
  if (a.wdtype == 0) e = nt == 1 ? launch_wt<0, 1>(p, pl.grid, st) : launch_wt<0, 2>(p, pl.grid, st);
  else if (a.wdtype == 1) e = nt == 1 ? launch_wt<1, 1>(p, pl.grid, st) : launch_wt<1, 2>(p, pl.grid, st);
  else e = nt == 1 ? launch_wt<2, 1>(p, pl.grid, st) : launch_wt<2, 2>(p, pl.grid, st);
  if (e != cudaSuccess) return fail_cuda(e);
  MOE_COUNT_LAUNCH();
  return MOE_OK;
}

}  // namespace moe

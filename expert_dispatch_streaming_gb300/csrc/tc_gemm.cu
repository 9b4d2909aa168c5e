// Grouped expert GEMM on the 5th-generation tensor cores (tcgen05 + TMEM), sm_103a.
//
// Computes, for every expert e that received rows [r0, r0 + n_e) of the permuted activations,
//   D[m][n] = sum_k W_e[m][k] * X[r0 + n][k]
// with W_e the expert's weight rows (gate and up rows for the first GEMM, down rows for the
// second) and X the token rows; the epilogue writes bf16(silu(gate) * up) (fused) or bf16(D).
// This is the grouped SwiGLU FFN of the MoE layer: only experts a batch selected are touched
// ("NovaLLM: Running Massive MoE Models Fully In-Memory", "3. Optimization #1 -- Expert-Level
// Streaming").
//
// Persistent kernel, one CTA per SM, warp-specialised:
//   warp 0      producer: per K step (64 wide; 128 for quantised weights), one 1-D bulk copy
//               per 128-row weight tile (the bundle stores each tile as its 128-byte-swizzled
//               shared-memory image; INT4 / NVFP4: the tile's codes and scales) and 2-D TMA
//               loads of the BN token rows (128-byte swizzle; quantised weights, a tile
//               that is not full: 32-row boxes of the rows present), completing on an mbarrier;
//   warp 1      MMA issuer: allocates TMEM, issues tcgen05.mma (M = 128 weight rows, N = BN
//               tokens, K = 16), commits stage release and accumulator-ready to mbarriers;
//   warps 2-5   epilogue: tcgen05.ld of the fp32 accumulators (each warp owns one 32-lane
//               quarter of TMEM), SiLU * mul, bf16 stores (or fp32 split-K partials);
//   warps 6-13  (INT4 / NVFP4) dequantisation: codes -> bf16(code * scale) written straight
//               into tensor memory with tcgen05.st; the MMA takes its A operand from there.
//               NVFP4's matrix scale multiplies the fp32 accumulator in the epilogue.
// Producer and MMA warps run their loops as whole, converged warps (warp-uniform descriptors,
// warp-vote waits) and issue from one lane chosen by elect.sync: a warp that waits in one
// divergent lane pays hundreds of cycles per step to reconverge, and an issue under a plain
// per-lane predicate keeps the MMA operands off the uniform datapath.
// Work unit = (expert with rows, 128-row weight tile, K split, BN token tile); units are
// enumerated with the token tile fastest so CTAs running at the same time share a weight
// tile through L2.  With split K, each split stores fp32 partials and the last CTA to finish
// a tile (one atomic counter, no waiting) sums the splits in order.
//
// Every mbarrier wait is bounded (wall clock, ~2 s); on timeout the kernel records an error
// word and leaves its loop, releasing TMEM before exit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "expert_ffn.cuh"
#include "tc_gemm.cuh"

namespace moe {

namespace {

constexpr uint64_t kWaitNs = 2000000000ull;

// Suspend-time hint (ns) of the mbarrier waits; 0 = plain polling.
#ifndef MOE_WAIT_HINT_NS
#define MOE_WAIT_HINT_NS 0
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
#if MOE_WAIT_HINT_NS > 0
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "n"(MOE_WAIT_HINT_NS)
      : "memory");
#else
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
#endif
  return ok != 0;
}
// Bounded wait of a whole converged warp: every lane polls and warp votes decide, so the warp
// never diverges (a divergent single-lane wait costs hundreds of cycles to reconverge).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int32_t* err, int code) {
  if (__all_sync(0xffffffffu, mbar_try(bar, parity))) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (__all_sync(0xffffffffu, mbar_try(bar, parity))) return true;
    if ((i & 255) == 0 && __any_sync(0xffffffffu, globaltimer() - t0 > kWaitNs)) {
      if ((threadIdx.x & 31) == 0) atomicExch(err, code);
      return false;
    }
  }
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
// One elected lane of a converged warp (elect.sync: the compiler can keep the issue path on
// the uniform datapath, which a plain lane test does not allow).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n.reg .pred p;\n.reg .b32 r;\nelect.sync r|p, 0xffffffff;\nselp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(pred));
  return pred != 0;
}
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                 // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset
  d |= (uint64_t)1 << 46;                 // descriptor version
  d |= (uint64_t)2 << 61;                 // 128-byte swizzle
  return d;
}
// Instruction descriptor of kind::f16: bf16 A and B, fp32 D, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
// tcgen05.mma of kind::f16 (bf16 A and B, fp32 accumulator in TMEM) from shared-memory
// descriptors, and (_ts) with the A operand in tensor memory (128 lanes = rows, two bf16 of K
// per column).
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16-column TMEM load without the wait (tcgen05.wait::ld follows before any use of r).
__device__ __forceinline__ void tmem_ld16_nw(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// Waits for this thread's TMEM loads; the loaded registers are tied to the wait so that no
// use of them is scheduled above it.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]),
        "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]),
        "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]),
        "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]),
        "+r"(b[11]), "+r"(b[12]), "+r"(b[13]), "+r"(b[14]), "+r"(b[15])
      :
      : "memory");
}

// Thread i of the warp writes registers r[0..N) into TMEM lane (taddr lane + i), columns
// taddr column .. +N-1 (the registers are read at issue); tcgen05.wait::st (tmem_wait_st)
// must follow before the data is handed to the MMA.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// silu(g) * u = g / (1 + e^-g) * u with the hardware exponential and reciprocal (relative error
// ~1e-6, far below the bf16 rounding of the result); for g below about -88, e^-g overflows
// to +inf and the quotient is -0, the limit of silu.
__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fdividef(g, 1.f + __expf(-g)) * u;
}

// Weight storage of a kernel variant: bf16 tile images, INT4 or NVFP4 tiles.
enum WType { kBf16 = 0, kInt4 = 1, kFp4 = 2 };

template <int BN, bool FUSED, int WT>
struct Cfg {
  static constexpr bool INT4 = WT != kBf16;                   // quantised: dequant warps
  static constexpr int NA = FUSED ? 2 : 1;                    // weight tiles per K step
  // K per pipeline step: 64 for bf16 (one 128 x 64 tile image); 128 for quantised weights,
  // one whole tile of 128 k (codes + its scales), which halves the per-step cost per FLOP
  static constexpr int KSTEP = INT4 ? 128 : 64;
  static constexpr int A_BYTES = 16384;                       // 128 rows x 64 k bf16
  static constexpr int B_SUB = BN * 128;                      // BN rows x 64 k bf16 (one box)
  static constexpr int B_BYTES = B_SUB * (KSTEP / 64);
  // one quantised tile per weight tile: INT4 8448 bytes, NVFP4 9216 bytes
  static constexpr int RAW_BYTES = WT == kInt4 ? 8448 : WT == kFp4 ? 9216 : 0;
  // shared-memory ring (filled by the producer): bf16 = A tile(s) + B tile; INT4 = B tiles +
  // raw INT4 tiles.  INT4 A tiles never touch shared memory: the dequant warps write them
  // into tensor memory (tcgen05.st) and the MMA reads A from there.
  static constexpr int R1 = INT4 ? (B_BYTES + NA * RAW_BYTES + 1023) / 1024 * 1024
                                 : NA * A_BYTES + B_BYTES;
  static constexpr int D1_FIT = (INT4 ? 220 : 200) * 1024 / R1;
  static constexpr int D1 = D1_FIT > 8 ? 8 : D1_FIT;
  static_assert(D1 >= 2, "the ring needs at least two stages");
  static constexpr int B_OFF = INT4 ? 0 : NA * A_BYTES;       // B tile inside a ring slot
  static constexpr int RAW_OFF = B_BYTES;                     // raw codes inside (INT4)
  static constexpr int TX = INT4 ? NA * RAW_BYTES + B_BYTES : NA * A_BYTES + B_BYTES;
  // tensor memory: accumulators (gate and up side by side when fused), double-buffered where
  // they fit, then (INT4) D2 stages of dequantised A, 64 columns (128 bf16 of K) per tile
  static constexpr int ACC = NA * BN;                         // TMEM columns per tile
  static constexpr int D2 = INT4 ? (FUSED ? 2 : 4) : 0;
  static constexpr int A_COLS = D2 * NA * (KSTEP / 2);
  static constexpr int BUFS = (2 * ACC + A_COLS <= 512) ? 2 : 1;
  static constexpr int A_TMEM = ACC * BUFS;                   // first column of the A stages
  static constexpr int USED = ACC * BUFS + A_COLS;
  static_assert(USED <= 512, "tensor memory holds 512 columns");
  static constexpr int TMEM_COLS = USED <= 32 ? 32 : USED <= 64 ? 64 : USED <= 128 ? 128
                                 : USED <= 256 ? 256 : 512;
  static constexpr int DQ_WARPS = 8;                          // quantised: dequant warps, 2 per quarter
  static constexpr int THREADS = INT4 ? 192 + 32 * DQ_WARPS : 192;
  static constexpr int SMEM = D1 * R1 + 1024 /*align*/ + 4096 /*barriers, prefix*/;
  static_assert(SMEM <= 232448, "over the 227 KB shared-memory limit of a CTA");
};

static_assert(sizeof(TcParams) <= 4096, "kernel parameters stay within 4 KB");

struct Unit {
  const char* w;            // weight section of this unit's expert
  const float* gs;          // NVFP4: the section's matrix scale(s) (gate, up or down)
  const CUtensorMap* tm;    // its token rows (tms: in 32-row boxes, quantised weights)
  const CUtensorMap* tms;
  uint16_t* out;
  float* part;
  int M, KT, MT, S, kps, max_rows;
  int r0, ne, mt, ks, nt, tile;
};

// Rows [r0, r0 + ne) of an expert as read from the offsets, clipped to the launch's
// [0, max_rows) so that offsets inconsistent with max_rows can never index past the buffers
// sized by it.  Returns true when the clip changed anything (the caller records error 8).
__device__ __forceinline__ bool clip_rows(int& r0, int& ne, int max_rows) {
  const int c0 = min(max(r0, 0), max_rows);
  const int cn = max(0, min(ne, max_rows - c0));
  const bool changed = c0 != r0 || cn != ne;
  r0 = c0;
  ne = cn;
  return changed;
}

// Maps unit index u to its (expert, row tile, split, token tile), from the per-expert prefix
// of unit counts kept in shared memory; units past the routed experts belong to the second
// group (the shared expert) when there is one.
__device__ __forceinline__ Unit decode_unit(const TcParams& p, const int* pref, int n_act,
                                            int u, int BN, int KSTEP) {
  Unit x;
  int base, tile_base;
  if (p.g2 && u >= pref[n_act]) {
    x.w = static_cast<const char*>(p.w2);
    x.gs = reinterpret_cast<const float*>(x.w + p.gs_rel2);
    x.tm = &p.tmap_b2;
    x.tms = &p.tmap_bs2;
    x.out = p.out2;
    x.part = p.part2;
    x.M = p.M2;
    x.KT = p.K2 / KSTEP;
    x.S = p.S2;
    x.kps = p.kt_per_split2;
    x.max_rows = p.rows2;
    x.r0 = 0;
    x.ne = p.rows2;
    base = pref[n_act];
    tile_base = pref[n_act] / p.S;
  } else {
    int lo = 0, hi = n_act - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pref[mid] <= u) lo = mid;
      else hi = mid - 1;
    }
    const int e = p.host_n >= 0 ? p.host_ids[lo] : p.active[lo];
    x.w = static_cast<const char*>(p.dev_tab ? p.dev_tab[e] : p.tab.p[e]) + p.w_off;
    x.gs = reinterpret_cast<const float*>(x.w + p.gs_rel);
    x.tm = &p.tmap_b;
    x.tms = &p.tmap_bs;
    x.out = p.out;
    x.part = p.part;
    x.M = p.M;
    x.KT = p.K / KSTEP;
    x.S = p.S;
    x.kps = p.kt_per_split;
    x.max_rows = p.max_rows;
    x.r0 = p.offsets[e];
    x.ne = p.offsets[e + 1] - x.r0;
    clip_rows(x.r0, x.ne, p.max_rows);
    base = pref[lo];
    tile_base = pref[lo] / p.S;
  }
  x.MT = x.M / 128;
  const int nt_n = (x.ne + BN - 1) / BN;
  int rem = u - base;
  x.nt = rem % nt_n;
  rem /= nt_n;
  x.ks = rem % x.S;
  x.mt = rem / x.S;
  x.tile = tile_base + x.mt * nt_n + x.nt;
  return x;
}

template <int BN, bool FUSED, int WT, bool ROUTER = false>
__global__ void __launch_bounds__(Cfg<BN, FUSED, WT>::THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ TcParams p) {
  using C = Cfg<BN, FUSED, WT>;
  constexpr bool INT4 = C::INT4;   // any quantised weight type
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::D1 * C::R1);
  uint64_t* full = bars;                    // ring 1: loaded
  uint64_t* empty = bars + 8;               // ring 1: consumed by the MMA
  uint64_t* afull = bars + 16;              // INT4: dequantised A stage in TMEM ready
  uint64_t* aempty = bars + 24;             // INT4: A stage consumed by the MMA
  uint64_t* tfull = bars + 32;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  int* pref = reinterpret_cast<int*>(tmem_slot + 4);   // [kMaxExperts + 2]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int MT = p.M / 128;
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int s = 0; s < 8; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
      mbar_init(smem_u32(&afull[s]), C::DQ_WARPS);
      mbar_init(smem_u32(&aempty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 4);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(C::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // everything above touches no memory that earlier kernels write; from here on the routing
  // results (offsets, expert list) and the token rows are read
  pdl_wait();
  const int n_act = p.host_n >= 0 ? p.host_n : *p.n_active;
  if (warp == 2) {
    // prefix of unit counts over the experts with rows
    int carry = 0;
    for (int base = 0; base < n_act; base += 32) {
      const int a = base + lane;
      int cnt = 0;
      if (a < n_act) {
        const int e = p.host_n >= 0 ? p.host_ids[a] : p.active[a];
        int r0 = p.offsets[e], ne = p.offsets[e + 1] - r0;
        if (clip_rows(r0, ne, p.max_rows)) atomicExch(p.err, 8);
        cnt = MT * p.S * ((ne + BN - 1) / BN);
      }
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (a < n_act) pref[a] = carry + incl - cnt;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      pref[n_act] = carry;
      pref[n_act + 1] = carry + (p.g2 ? (p.M2 / 128) * p.S2 * ((p.rows2 + BN - 1) / BN) : 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = pref[n_act + 1];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop (warp-uniform addresses, converged waits); one elected lane
    // issues the copies.
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const Unit x = decode_unit(p, pref, n_act, u, BN, C::KSTEP);
      const char* wb = x.w;
      const int KT = x.KT, MTx = x.MT;
      const int kt_lo = x.ks * x.kps, kt_hi = min(KT, kt_lo + x.kps);
      for (int kt = kt_lo; kt < kt_hi; ++kt) {
        if (!(ok = warp_wait(smem_u32(&empty[stage]), phase ^ 1, p.err, 1))) break;
        const uint32_t fb = smem_u32(&full[stage]);
        uint8_t* st = smem + stage * C::R1;
        // token rows: one box of BN rows; quantised kernels load a tile that is not full in
        // boxes of 32 rows, only those of the rows present
        const int nsub = INT4 && x.ne - x.nt * BN < BN ? (x.ne - x.nt * BN + 31) >> 5 : 0;
        if (elect_one()) {
          mbar_expect_tx(fb, nsub ? C::NA * C::RAW_BYTES + (C::KSTEP / 64) * nsub * 4096 : C::TX);
          if (INT4) {
            // the whole 128-k quantised tile (codes + row scales) of each weight tile
#pragma unroll
            for (int w = 0; w < C::NA; ++w)
              bulk_g2s(smem_u32(st + C::RAW_OFF + w * C::RAW_BYTES),
                       wb + ((size_t)(x.mt + w * MTx) * KT + kt) * C::RAW_BYTES, C::RAW_BYTES,
                       fb);
          } else {
            bulk_g2s(smem_u32(st), wb + ((size_t)x.mt * KT + kt) * C::A_BYTES,
                        C::A_BYTES, fb);
            if (FUSED)
              bulk_g2s(smem_u32(st + C::A_BYTES),
                          wb + ((size_t)(x.mt + MTx) * KT + kt) * C::A_BYTES, C::A_BYTES, fb);
          }
#pragma unroll
          for (int b = 0; b < C::KSTEP / 64; ++b) {
            const int kc = (ROUTER ? kt % p.kb_mod : kt) * C::KSTEP + b * 64;
            if (nsub) {
              // 32-row boxes of 4 KB stacked at 4 KB steps: the same 128-byte-swizzled layout
              // as one box of all the rows (the swizzle follows the address bits)
              for (int sb = 0; sb < nsub; ++sb)
                tma_2d(smem_u32(st + C::B_OFF + b * C::B_SUB + sb * 4096), x.tms, kc,
                       x.r0 + x.nt * BN + 32 * sb, fb);
            } else {
              tma_2d(smem_u32(st + C::B_OFF + b * C::B_SUB), x.tm, kc, x.r0 + x.nt * BN, fb);
            }
          }
        }
        __syncwarp();
        if (++stage == C::D1) { stage = 0; phase ^= 1; }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // As the producer: the converged warp computes the descriptors, one elected lane issues.
    int stage = 0, buf = 0, astage = 0;
    uint32_t phase = 0, aphase = 0, a2phase = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const Unit x = decode_unit(p, pref, n_act, u, BN, C::KSTEP);
      const int kt_lo = x.ks * x.kps, kt_hi = min(x.KT, kt_lo + x.kps);
      // the last token tile of a group is ragged: multiply only its first N = n_here rounded
      // up to 16 columns (the accumulator columns past it are never read)
      const int n_here = min(BN, x.ne - x.nt * BN);
      const uint32_t idesc = idesc_bf16(128, min(BN, (n_here + 15) & ~15));
      if (!(ok = warp_wait(smem_u32(&tempty[buf]), aphase ^ 1, p.err, 2))) break;
      const uint32_t dg = tmem_base + buf * C::ACC;
      for (int kt = kt_lo; kt < kt_hi; ++kt) {
        // INT4: the dequant warps arrive on afull only after they saw this stage's full
        // barrier, so afull alone orders the B tile as well
        if (!INT4 && !(ok = warp_wait(smem_u32(&full[stage]), phase, p.err, 3))) break;
        if (INT4 && !(ok = warp_wait(smem_u32(&afull[astage]), a2phase, p.err, 6))) break;
        const uint32_t s1 = smem_u32(smem + stage * C::R1);
        const uint64_t db = sdesc_sw128(s1 + C::B_OFF);
        if (elect_one()) {
          tc_fence_after();
          if (INT4) {
            // A from tensor memory: tile w of this stage at columns A_TMEM + (astage*NA + w)*64,
            // eight columns (16 k) per MMA; B from the step's two 64-k boxes
            const uint32_t ta = tmem_base + C::A_TMEM + astage * C::NA * 64;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t acc = (kt > kt_lo || j > 0) ? 1u : 0u;
              const uint64_t bj = sdesc_sw128(s1 + C::B_OFF + (j >> 2) * C::B_SUB) + 2 * (j & 3);
              mma_bf16_ts(dg, ta + 8 * j, bj, idesc, acc);
              if (FUSED) mma_bf16_ts(dg + BN, ta + 64 + 8 * j, bj, idesc, acc);
            }
          } else {
            const uint64_t da = sdesc_sw128(s1), du = sdesc_sw128(s1 + C::A_BYTES);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t acc = (kt > kt_lo || j > 0) ? 1u : 0u;
              mma_bf16(dg, da + 2 * j, db + 2 * j, idesc, acc);
              if (FUSED) mma_bf16(dg + BN, du + 2 * j, db + 2 * j, idesc, acc);
            }
          }
          mma_commit(smem_u32(&empty[stage]));
          if (INT4) mma_commit(smem_u32(&aempty[astage]));
        }
        __syncwarp();
        if (++stage == C::D1) { stage = 0; phase ^= 1; }
        if (INT4 && ++astage == C::D2) { astage = 0; a2phase ^= 1; }
      }
      if (!ok) break;
      if (elect_one()) mma_commit(smem_u32(&tfull[buf]));
      __syncwarp();
      if (++buf == C::BUFS) { buf = 0; aphase ^= 1; }
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;                       // TMEM lane quarter of this warp
    const int et = threadIdx.x - 64;              // 0..127
    int buf = 0;
    uint32_t aphase = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const Unit x = decode_unit(p, pref, n_act, u, BN, C::KSTEP);
      const int MP = FUSED ? 2 * x.M : x.M;
      // NVFP4: the accumulators hold sum(E2M1 * scale * 2^-7 * x); times matrix scale * 2^7
      float gsc = 1.f, usc = 1.f;
      if (WT == kFp4) {
        gsc = __ldg(x.gs) * 128.f;
        if (FUSED) usc = __ldg(x.gs + 1) * 128.f;
      }
      if (!(ok = warp_wait(smem_u32(&tfull[buf]), aphase, p.err, 4))) break;
      tc_fence_after();
      const int m = x.mt * 128 + q * 32 + lane;
      const int n_here = min(BN, x.ne - x.nt * BN);
      const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16) + buf * C::ACC;
      // columns per TMEM load: 32, or 16 in the quantised kernels (more warps, fewer registers)
      constexpr int CH = INT4 ? 16 : 32;
      // write-out of columns c0 .. c0 + CH - 1 (bf16 h / y, fp32 partials, or router logits)
      // from the registers g (and v: the up accumulator)
      auto emit = [&](int c0, const uint32_t* g, const uint32_t* v) {
#pragma unroll
        for (int j = 0; j < CH; ++j) {
          const int n = c0 + j;
          if (n < n_here) {
            const size_t row = (size_t)(x.r0 + x.nt * BN + n);
            const float gv = __uint_as_float(g[j]) * gsc;
            if (ROUTER && x.S == 1) {
              if (m < p.m_limit) p.out_f32[row * p.ldo + m] = gv;
            } else if (x.S == 1) {
              const float o = FUSED ? silu_mul(gv, __uint_as_float(v[j]) * usc) : gv;
              x.out[row * x.M + m] = float_to_bf16_bits(o);
            } else {
              float* pr = x.part + ((size_t)x.ks * x.max_rows + row) * MP;
              pr[m] = gv;
              if (FUSED) pr[x.M + m] = __uint_as_float(v[j]) * usc;
            }
          }
        }
      };
      if constexpr (INT4) {
        // quantised kernels (16-column chunks): the next chunk's TMEM loads are in flight
        // while this chunk is written out; the accumulator buffer is single here, so the
        // epilogue is on the MMA's critical path
        const int nch = (n_here + CH - 1) / CH;   // warp-uniform
        uint32_t gA[CH], vA[CH], gB[CH], vB[CH];
#pragma unroll
        for (int j = 0; j < CH; ++j) vA[j] = vB[j] = 0u;
        tmem_ld16_nw(ta, gA);
        if (FUSED) tmem_ld16_nw(ta + BN, vA);
        tmem_wait_ld(gA, vA);
#pragma unroll 1
        for (int c = 0; c < nch; c += 2) {
          if (c + 1 < nch) {
            tmem_ld16_nw(ta + (c + 1) * CH, gB);
            if (FUSED) tmem_ld16_nw(ta + BN + (c + 1) * CH, vB);
          }
          emit(c * CH, gA, vA);
          if (c + 1 >= nch) break;
          tmem_wait_ld(gB, vB);
          if (c + 2 < nch) {
            tmem_ld16_nw(ta + (c + 2) * CH, gA);
            if (FUSED) tmem_ld16_nw(ta + BN + (c + 2) * CH, vA);
          }
          emit((c + 1) * CH, gB, vB);
          tmem_wait_ld(gA, vA);
        }
      } else {
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += CH) {
          if (c0 >= n_here) break;   // warp-uniform
          uint32_t g[CH], v[CH];
          tmem_ld32(ta + c0, g);
          if (FUSED) tmem_ld32(ta + BN + c0, v);
          emit(c0, g, v);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty[buf]));
      if (++buf == C::BUFS) { buf = 0; aphase ^= 1; }

      if (!ROUTER && x.S > 1) {
        // per (tile, lane quarter) arrival counter: the warp completing the S arrivals of its
        // quarter sums that quarter's 32 rows over the splits in split order (no barrier,
        // nothing waits, the four quarters reduce in parallel).  The router's split partials
        // are summed by its consumer, the gating kernel.
        __threadfence();
        __syncwarp();
        int last = 0;
        int32_t* ctr = p.counters + (size_t)x.tile * 4 + q;
        if (lane == 0) {
          const int prev = atomicAdd(ctr, 1);
          last = prev == x.S - 1;
          if (last) *ctr = 0;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();
          const size_t stride = (size_t)x.max_rows * MP;
          for (int n = 0; n < n_here; ++n) {
            const size_t row = (size_t)(x.r0 + x.nt * BN + n);
            const float* pr = x.part + row * MP + m;
            // four interleaved running sums keep four split loads in flight; fixed order
            float g0 = 0.f, g1 = 0.f, g2 = 0.f, g3 = 0.f, u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
            int sp = 0;
            for (; sp + 4 <= x.S; sp += 4) {
              g0 += __ldcg(pr + sp * stride);
              g1 += __ldcg(pr + (sp + 1) * stride);
              g2 += __ldcg(pr + (sp + 2) * stride);
              g3 += __ldcg(pr + (sp + 3) * stride);
              if (FUSED) {
                u0 += __ldcg(pr + x.M + sp * stride);
                u1 += __ldcg(pr + x.M + (sp + 1) * stride);
                u2 += __ldcg(pr + x.M + (sp + 2) * stride);
                u3 += __ldcg(pr + x.M + (sp + 3) * stride);
              }
            }
            for (; sp < x.S; ++sp) {
              g0 += __ldcg(pr + sp * stride);
              if (FUSED) u0 += __ldcg(pr + x.M + sp * stride);
            }
            const float gs = (g0 + g1) + (g2 + g3), us = (u0 + u1) + (u2 + u3);
            x.out[row * x.M + m] = float_to_bf16_bits(FUSED ? silu_mul(gs, us) : gs);
          }
        }
      }
    }
    (void)et;
  } else if (INT4) {
    // ------------------------------------------------------------ dequant (warps 6 ..)
    // A warp may only touch its own quarter of the TMEM lanes (warp % 4), so DQ_WARPS / 4 warps
    // share each quarter: thread = weight row r = 32 * (warp % 4) + lane, and the warp's job
    // (its rank among its quarter's warps) is CPW consecutive 32-code chunks of the step's
    // NA * 4 (the row's 128 codes of each weight tile), all in one tile: 16 TMEM columns per
    // chunk, pairs in k order.  Fused: the gate tile's 4 chunks, or the up tile's; not fused:
    // chunks 0-1 or 2-3.  (Sixteen dequant warps, one pair of chunks each, measured no faster
    // for the fused GEMMs and slower for the down GEMMs, at the 80 registers a thread they allow.)
    constexpr int JOBS = C::DQ_WARPS / 4, CPW = C::NA * 4 / JOBS;
    static_assert(CPW == 2 || CPW == 4, "whole pairs of chunks of one tile");
    const int q = warp & 3, job = (warp - 6) >> 2, r = q * 32 + lane;
    const int tile = job * CPW / 4, c_lo = job * CPW % 4;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int stage = 0, astage = 0;
    uint32_t phase = 0, a2phase = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const Unit x = decode_unit(p, pref, n_act, u, BN, C::KSTEP);
      const int kt_lo = x.ks * x.kps, kt_hi = min(x.KT, kt_lo + x.kps);
      for (int kt = kt_lo; kt < kt_hi; ++kt) {
        if (!(ok = warp_wait(smem_u32(&full[stage]), phase, p.err, 5))) break;
        if (!(ok = warp_wait(smem_u32(&aempty[astage]), a2phase ^ 1, p.err, 7))) break;
        tc_fence_after();
        const uint8_t* raw = smem + stage * C::R1 + C::RAW_OFF + tile * C::RAW_BYTES;
        // INT4: one bf16 group scale per row and tile; NVFP4: eight E4M3 block scales (16 k)
        uint32_t s2 = 0;
        uint2 s8 = make_uint2(0, 0);
        if (WT == kInt4) s2 = int4_scale_pair(*reinterpret_cast<const uint16_t*>(raw + 8192 + 2 * r));
        else s8 = *reinterpret_cast<const uint2*>(raw + 8192 + 8 * r);
        const uint32_t ta = tmem_base + lane_base + C::A_TMEM + (astage * C::NA + tile) * 64;
        // chunks c0 .. c0 + NCH - 1 of row r -> TMEM columns 16 c0 .. 16 (c0 + NCH) - 1
        auto convert = [&](auto nch, int c0) {
          constexpr int NCH = decltype(nch)::value;
          uint32_t w[4 * NCH];
#pragma unroll
          for (int i = 0; i < NCH; ++i) {
            const uint4 a = *reinterpret_cast<const uint4*>(raw + ((c0 + i) * 128 + r) * 16);
            w[4 * i] = a.x;
            w[4 * i + 1] = a.y;
            w[4 * i + 2] = a.z;
            w[4 * i + 3] = a.w;
          }
          uint32_t v[16 * NCH];
#pragma unroll
          for (int jp = 0; jp < 2 * NCH; ++jp) {
            // words 2 jp, 2 jp + 1 (16 k) of chunk c = c0 + jp / 2 share one scale: NVFP4 block
            // 2 c + jp % 2 of the row, byte 2 (c % 2) + jp % 2 of the scale word of blocks
            // 4 (c / 2) .. 4 (c / 2) + 3
            uint32_t sp = s2;
            if (WT != kInt4) {
              const int c = c0 + jp / 2;
              sp = fp4_scale_pair(c < 2 ? s8.x : s8.y, 2 * (c & 1) + (jp & 1));
            }
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              const int j = 2 * jp + jj;
              if (WT == kInt4) {
                v[4 * j + 0] = int4_pair<0>(w[j], sp);
                v[4 * j + 1] = int4_pair<1>(w[j], sp);
                v[4 * j + 2] = int4_pair<2>(w[j], sp);
                v[4 * j + 3] = int4_pair<3>(w[j], sp);
              } else {
                v[4 * j + 0] = fp4_pair<0>(w[j], sp);
                v[4 * j + 1] = fp4_pair<1>(w[j], sp);
                v[4 * j + 2] = fp4_pair<2>(w[j], sp);
                v[4 * j + 3] = fp4_pair<3>(w[j], sp);
              }
            }
          }
          tmem_st32(ta + 16 * c0, v);
        };
        if constexpr (CPW == 4) {
          convert(std::integral_constant<int, 2>{}, 0);
          convert(std::integral_constant<int, 2>{}, 2);
        } else {
          convert(std::integral_constant<int, 2>{}, c_lo);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&afull[astage]));
        if (++stage == C::D1) { stage = 0; phase ^= 1; }
        if (++astage == C::D2) { astage = 0; a2phase ^= 1; }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(C::TMEM_COLS));
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

template <int BN, bool FUSED, int WT, bool ROUTER = false>
int launch_bn(TcParams& kp, cudaStream_t st) {
  using C = Cfg<BN, FUSED, WT>;
  static bool attr = false;
  if (!attr) {
    MOE_CUDA_TRY(cudaFuncSetAttribute(tc_gemm_kernel<BN, FUSED, WT, ROUTER>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
    attr = true;
  }
  MOE_LAUNCH_PDL(tc_gemm_kernel<BN, FUSED, WT, ROUTER>, dim3(sm_count()), dim3(C::THREADS),
                 C::SMEM, st, kp);
  MOE_COUNT_LAUNCH();
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

template <int WT>
int dispatch_bn(bool fused, int BN, TcParams& kp, cudaStream_t st) {
  if (fused) {
    switch (BN) {
      case 32: return launch_bn<32, true, WT>(kp, st);
      case 64: return launch_bn<64, true, WT>(kp, st);
      case 128: return launch_bn<128, true, WT>(kp, st);
      default:
        // quantised gate/up tiles stop at 128 tokens: their accumulators share tensor memory
        // with the dequantised weight stages
        if constexpr (WT != kBf16) return launch_bn<128, true, WT>(kp, st);
        else return launch_bn<256, true, WT>(kp, st);
    }
  }
  switch (BN) {
    case 32: return launch_bn<32, false, WT>(kp, st);
    case 64: return launch_bn<64, false, WT>(kp, st);
    case 128: return launch_bn<128, false, WT>(kp, st);
    default:
      if constexpr (WT != kBf16) return launch_bn<128, false, WT>(kp, st);
      else return launch_bn<256, false, WT>(kp, st);
  }
}

int dispatch_wt(const GemmArgs& a, int BN, TcParams& kp, cudaStream_t st) {
  if (a.fp4) return dispatch_bn<kFp4>(a.fused, BN, kp, st);
  if (a.int4) return dispatch_bn<kInt4>(a.fused, BN, kp, st);
  return dispatch_bn<kBf16>(a.fused, BN, kp, st);
}

}  // namespace

bool tc_supported(const GemmArgs& a) { return a.K % 128 == 0 && a.M % 128 == 0; }

int tc_bn_for(const GemmArgs& a) {
  const int A = std::max(1, a.host_n >= 0 ? std::min(a.host_n, a.max_rows)
                                          : std::min(a.E, a.max_rows));
  const int avg = ceil_div(std::max(a.max_rows, 1), A);
  // fused tiles hold gate and up accumulators: a 256-token tile would fill all of TMEM (no
  // double buffer, the epilogue not overlapped with the next tile's MMA; with INT4 no room for
  // the dequantised weight stages); 128-token fused tiles measured faster at every bf16 shape
  // INT4 down tiles also stop at 128 tokens: at 256 the accumulator and the dequantised A
  // stages fill TMEM without a second accumulator buffer, so the epilogue would not overlap
  const int cap = (a.fused || a.int4 || a.fp4) ? 128 : 256;
  int bn = avg <= 32 ? 32 : avg <= 64 ? 64 : avg <= 128 ? 128 : 256;
  if (a.int4 || a.fp4) {
    // quantised weights are decoded once per token tile, so the tile is as wide as the most
    // rows one expert can hold (a skewed batch puts most of its tokens on a few experts);
    // its MMAs and token-row loads cover only the rows present, so a wide tile costs an
    // expert with few rows nothing but the second accumulator buffer
    const int most = a.rows_cap > 0 ? std::min(a.rows_cap, a.max_rows) : a.max_rows;
    bn = std::max(bn, most <= 32 ? 32 : most <= 64 ? 64 : 128);
  }
  return std::min(bn, cap);
}

TcPlan plan_tc(const GemmArgs& a) {
  TcPlan t{};
  t.BN = tc_bn_for(a);
  const int A = std::max(1, a.host_n >= 0 ? std::min(a.host_n, a.max_rows)
                                          : std::min(a.E, a.max_rows));
  const bool q = a.int4 || a.fp4;
  const int MT = a.M / 128, KT = a.K / (q ? 128 : 64), sms = sm_count();
  const int avg = ceil_div(std::max(a.max_rows, 1), A);
  // narrower token tiles first (more tiles, weights re-read from L2 only), then split K
  while (t.BN > 32 && A * MT * ceil_div(avg, t.BN) < sms &&
         ceil_div(avg, t.BN / 2) > ceil_div(avg, t.BN))
    t.BN /= 2;
  const int ntiles_est = A * MT * std::max(1, ceil_div(avg, t.BN));
  // split K so that the units fill whole waves of the persistent grid: the time of a launch
  // is ~ ceil(units / SMs) waves of 1/S of the K range each; fp32 partial traffic caps S
  const double wbytes =
      (double)A * MT * 128 * a.K * (a.fp4 ? 0.56 : a.int4 ? 0.52 : 2.0) * (a.fused ? 2 : 1);
  const double pbytes = (double)a.max_rows * (a.fused ? 2 : 1) * a.M * 8.0;
  const int s_cap = std::min(KT, std::max(1, (int)(wbytes / std::max(pbytes, 1.0) / 4)));
  int S = 1;
  double best = (double)ceil_div(ntiles_est, sms);
  for (int s = 2; ntiles_est < sms && s <= std::min(s_cap, 32); ++s) {
    const double cost = (double)ceil_div(ntiles_est * s, sms) / s * (1.0 + 0.02 * (s - 1));
    if (cost < best * 0.97) {
      best = cost;
      S = s;
    }
  }
  t.kt_per_split = ceil_div(KT, S);
  t.S = ceil_div(KT, t.kt_per_split);
  const size_t mp = (size_t)(a.fused ? 2 : 1) * a.M;
  t.part_elems = t.S > 1 ? (size_t)t.S * a.max_rows * mp : 0;
  t.counter_elems = 4 * ((size_t)MT * (ceil_div(a.max_rows, t.BN) + A) + 1);
  return t;
}

static bool encode_tokens(CUtensorMap* m, const uint16_t* base, int K, int rows, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int fill_params(TcParams& kp, const GemmArgs& a, const TcPlan& t, float* part,
                       int32_t* counters, int32_t* err) {
  if (!encode_fn()) return MOE_ERR_UNSUPPORTED;
  if (!encode_tokens(&kp.tmap_b, a.xin, a.K, a.max_rows, t.BN)) return MOE_ERR_INVALID_ARG;
  if ((a.int4 || a.fp4) && !encode_tokens(&kp.tmap_bs, a.xin, a.K, a.max_rows, 32))
    return MOE_ERR_INVALID_ARG;
  kp.offsets = a.offsets;
  kp.active = a.active;
  kp.n_active = a.n_active;
  kp.host_n = a.host_n;
  for (int i = 0; i < (a.host_n > 0 ? a.host_n : 0); ++i) kp.host_ids[i] = (int16_t)a.host_ids[i];
  kp.tab = *a.tab;
  kp.dev_tab = a.dev_tab;
  kp.w_off = a.w_off;
  kp.gs_rel = a.gs_rel;
  kp.K = a.K;
  kp.M = a.M;
  kp.S = t.S;
  kp.kt_per_split = t.kt_per_split;
  kp.max_rows = a.max_rows;
  kp.out = a.out;
  kp.part = part;
  kp.counters = counters;
  kp.err = err;
  return MOE_OK;
}

int launch_tc(const GemmArgs& a, const TcPlan& t, float* part, int32_t* counters, int32_t* err,
              cudaStream_t st) {
  if (a.max_rows <= 0 || a.host_n == 0) return MOE_OK;
  TcParams kp{};
  const int r = fill_params(kp, a, t, part, counters, err);
  if (r != MOE_OK) return r;
  return dispatch_wt(a, t.BN, kp, st);
}

TcPair plan_tc_pair(const GemmArgs& a1, const GemmArgs& a2) {
  TcPair pp;
  pp.t1 = plan_tc(a1);
  pp.t2 = pp.t1;
  const int BN = pp.t1.BN, sms = sm_count();
  // tile counts of both groups at the routed group's token-tile width; one split count for
  // both, chosen on the combined tile count like plan_tc does for one group
  const int A = std::max(1, a1.host_n >= 0 ? std::min(a1.host_n, a1.max_rows)
                                           : std::min(a1.E, a1.max_rows));
  const int avg = ceil_div(std::max(a1.max_rows, 1), A);
  const int kstep = (a1.int4 || a1.fp4) ? 128 : 64;
  const int KT1 = a1.K / kstep, KT2 = a2.K / kstep;
  const int nt1 = A * (a1.M / 128) * std::max(1, ceil_div(avg, BN));
  const int nt2 = (a2.M / 128) * ceil_div(std::max(a2.max_rows, 1), BN);
  const int nt = nt1 + nt2;
  const double wb = ((double)A * a1.M * a1.K + (double)a2.M * a2.K) *
                    (a1.fp4 ? 0.56 : a1.int4 ? 0.52 : 2.0) * (a1.fused ? 2 : 1);
  const double pb = ((double)a1.max_rows * a1.M + (double)a2.max_rows * a2.M) *
                    (a1.fused ? 2 : 1) * 8.0;
  const int s_cap = std::min({KT1, KT2, std::max(1, (int)(wb / std::max(pb, 1.0) / 4))});
  int S = 1;
  double best = (double)ceil_div(nt, sms);
  for (int sp = 2; nt < sms && sp <= std::min(s_cap, 32); ++sp) {
    const double cost = (double)ceil_div(nt * sp, sms) / sp * (1.0 + 0.02 * (sp - 1));
    if (cost < best * 0.97) {
      best = cost;
      S = sp;
    }
  }
  pp.t1.kt_per_split = ceil_div(KT1, S);
  pp.t1.S = ceil_div(KT1, pp.t1.kt_per_split);
  pp.t2.kt_per_split = ceil_div(KT2, S);
  pp.t2.S = ceil_div(KT2, pp.t2.kt_per_split);
  const size_t mp1 = (size_t)(a1.fused ? 2 : 1) * a1.M, mp2 = (size_t)(a2.fused ? 2 : 1) * a2.M;
  pp.t1.part_elems = pp.t1.S > 1 ? (size_t)pp.t1.S * a1.max_rows * mp1 : 0;
  pp.t2.part_elems = pp.t2.S > 1 ? (size_t)pp.t2.S * a2.max_rows * mp2 : 0;
  pp.t1.counter_elems = 4 * ((size_t)(a1.M / 128) * (ceil_div(a1.max_rows, BN) + A) + nt2 + 1);
  return pp;
}

int launch_tc_pair(const GemmArgs& a1, const GemmArgs& a2, const TcPair& pp, float* part1,
                   float* part2, int32_t* counters, int32_t* err, cudaStream_t st) {
  if (a1.max_rows <= 0) return launch_tc(a2, pp.t2, part2, counters, err, st);
  TcParams kp{};
  int r = fill_params(kp, a1, pp.t1, part1, counters, err);
  if (r != MOE_OK) return r;
  if (a2.max_rows > 0) {
    if (!encode_tokens(&kp.tmap_b2, a2.xin, a2.K, a2.max_rows, pp.t1.BN) ||
        ((a1.int4 || a1.fp4) && !encode_tokens(&kp.tmap_bs2, a2.xin, a2.K, a2.max_rows, 32)))
      return MOE_ERR_INVALID_ARG;
    kp.g2 = 1;
    kp.w2 = static_cast<const char*>(a2.tab->p[0]) + a2.w_off;
    kp.gs_rel2 = a2.gs_rel;
    kp.M2 = a2.M;
    kp.K2 = a2.K;
    kp.S2 = pp.t2.S;
    kp.kt_per_split2 = pp.t2.kt_per_split;
    kp.rows2 = a2.max_rows;
    kp.out2 = a2.out;
    kp.part2 = part2;
  }
  return dispatch_wt(a1, pp.t1.BN, kp, st);
}

int tc_router_splits(int T, int H, int Mpad) {
  // K splits of the router product: its tiles (Mpad / 128 x ceil(T / 128)) are few next to the
  // SMs except at the largest batches.  Same rule as the expert GEMMs' split choice: the
  // fewest waves of 1/S of the K range each, a little extra per split (its partials, which the
  // gating kernel sums), at most 16 splits and at least 8 K steps per split.
  const int tiles = (Mpad / 128) * ceil_div(T, 128), KT = 3 * H / 64, G = sm_count();
  int best_s = 1;
  double best = (double)ceil_div(tiles, G);
  for (int S = 2; S <= std::min(16, KT / 8); ++S) {
    const double c = (double)ceil_div(tiles * S, G) / S * (1.0 + 0.05 * (S - 1));
    if (c < best * 0.97) {
      best = c;
      best_s = S;
    }
  }
  return ceil_div(KT, ceil_div(KT, best_s));
}

int launch_tc_router(const uint16_t* x, int T, int H, const void* img, int Mpad, int C,
                     const int32_t* meta, float* logits, float* part, int32_t* err,
                     cudaStream_t st) {
  if (T <= 0) return MOE_OK;
  auto enc = encode_fn();
  if (!enc) return MOE_ERR_UNSUPPORTED;
  constexpr int BN = 128;
  TcParams kp{};
  cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[1] = {(cuuint64_t)H * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)BN};
  cuuint32_t estr[2] = {1, 1};
  if (enc(&kp.tmap_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims,
          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MOE_ERR_INVALID_ARG;
  kp.offsets = meta;
  kp.active = meta + 2;
  kp.n_active = meta + 3;
  kp.host_n = -1;
  kp.tab.p[0] = img;
  kp.w_off = 0;
  kp.K = 3 * H;
  kp.M = Mpad;
  kp.S = tc_router_splits(T, H, Mpad);
  kp.kt_per_split = ceil_div(3 * H / 64, kp.S);
  kp.part = part;          // [S][T][Mpad] fp32 when S > 1
  kp.max_rows = T;
  kp.err = err;
  kp.kb_mod = H / 64;
  kp.out_f32 = logits;
  kp.ldo = C;
  kp.m_limit = C;
  return launch_bn<BN, false, kBf16, true>(kp, st);
}

}  // namespace moe

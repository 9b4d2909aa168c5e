/*
 * moe.h -- C ABI of libmoe: the Mixture-of-Experts layer forward with an expert-slot cache,
 * for NVIDIA GB300 (sm_103a).
 *
 * The layer (pages: "NovaLLM: Running Massive MoE Models Fully In-Memory", sections
 * "2. Why MoE Is a Natural Breakthrough Point" and "3. Optimization #1 -- Expert-Level
 * Streaming"; "Running 35B MoE Models on 8GB GPUs: How vvllm-ms Caches Experts in System
 * RAM", section "Technical Insight") runs, per call:
 *
 *   router logits -> top-k gating -> per-expert histogram + prefix scan -> permutation into
 *   expert-contiguous order -> grouped SwiGLU expert FFN -> gate-weighted combine,
 *
 * fed, when a cache is attached, by fixed VRAM slots that hold expert bundles copied on
 * demand from pinned host memory under LRU eviction.
 *
 * Conventions (every entry point):
 *  - Returns an int status: MOE_OK (0) or a negative MOE_ERR_* code.  No C++ exception
 *    crosses this boundary.  After MOE_ERR_CUDA, moe_last_cuda_error() returns the
 *    cudaError_t value that caused it.
 *  - The caller owns every device and host buffer passed in (allocated however it likes);
 *    the library never frees them.  Scratch memory is a caller-provided device buffer `ws`
 *    of at least the bytes reported by the matching *_workspace_size() query; its contents
 *    on entry do not matter and it must not be shared by calls that overlap on the GPU.
 *    The only objects the library allocates are expert caches (moe_expert_cache_*).
 *  - Device work is enqueued on the caller's CUDA stream `stream` (a cudaStream_t passed
 *    as void*; NULL = the legacy default stream) and the call returns without waiting,
 *    except where a function says it waits.
 *  - Pointers documented "device" must be device-accessible global memory; "host" are
 *    ordinary host pointers.  Device buffers must be 16-byte aligned; row strides are the
 *    row lengths stated (dense, row-major).
 *  - bf16 values are passed as uint16_t bit patterns.  INT4 weights are passed as int8 codes
 *    in [-7, 7]; NVFP4 weights as one FP4 E2M1 code per byte and one FP8 E4M3 byte per block
 *    scale (see moe_pack_bundle and moe_pack_bundle_nvfp4).
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ status codes */
enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1, /* a null pointer, bad size, unsupported shape or misalignment */
  MOE_ERR_CUDA = -2,        /* a CUDA runtime call failed; see moe_last_cuda_error()       */
  MOE_ERR_CAPACITY = -3,    /* a cache request needs more distinct bundles than slots      */
  MOE_ERR_TIMEOUT = -4,     /* a bounded host wait on GPU work ran out of time             */
  MOE_ERR_CORRUPT = -5,     /* a host bundle failed its checksum at cache creation         */
  MOE_ERR_UNSUPPORTED = -6, /* valid request this build does not implement                 */
  MOE_ERR_NO_MEMORY = -7    /* the cache could not allocate its VRAM slots or events       */
};

/* The cudaError_t value of the last MOE_ERR_CUDA on this thread (0 if none). */
int moe_last_cuda_error(void);
/* A static string naming a status code. */
const char* moe_status_string(int status);
/* Library version, (major << 16) | minor. */
int moe_version(void);

/* Process-wide options (set before enqueueing work; not thread-safe).
 *  MOE_OPT_FFN_KERNEL: which expert-FFN kernel runs: 0 = automatic (default: the tensor-core
 *    tcgen05 kernel wherever it supports the weight type, else the mma.sync weight-streaming
 *    kernel), 1 = always the streaming kernel, 2 = tcgen05 wherever supported.  Both compute
 *    the same layer; tests use the option to cover both.
 *  MOE_OPT_PDL: 1 = launch the layer's kernels with programmatic dependent launch (a kernel
 *    is scheduled while its predecessor finishes and waits in-kernel for its results); 0
 *    (default) = plain stream-ordered launches, which measured as fast or faster on GB300 at
 *    every workload tried.  Results are identical either way.
 *  MOE_OPT_DECODE_KERNEL: 2 = moe_layer_forward runs a batch of at most 16 tokens with every
 *    bundle resident (no cache) as one cooperative launch that routes, runs the shared and
 *    routed experts and combines; 1 (default) = the same except for INT4 weights with more
 *    than 4 tokens, which take the step-by-step kernels (faster for them there on GB300);
 *    0 = always the step-by-step kernels.  Both compute the same layer (same roundings; sums in a different
 *    fixed order). */
enum moe_option { MOE_OPT_FFN_KERNEL = 1, MOE_OPT_PDL = 2, MOE_OPT_DECODE_KERNEL = 3 };
int moe_set_option(int option, int value);

/* Reads the device error word kept in the first 4 bytes of a moe_layer_forward,
 * moe_grouped_swiglu or moe_route_topk workspace into *code (host) and waits for `stream`.
 * 0 = no error; otherwise the last call on that workspace produced invalid outputs:
 *   1-7  a bounded wait inside a tensor-core kernel ran out of time;
 *   9    a bounded wait inside the fused decode kernel ran out of time;
 *   8    an expert's row range [offsets[e], offsets[e+1]) reached outside [0, max_rows)
 *        (moe_grouped_swiglu) and was clipped to it;
 *   20   a device-LRU cache request needed more distinct bundles than slots.
 * Blocking (test and debug use). */
int moe_workspace_error(const void* ws, int32_t* code, void* stream);

/* ------------------------------------------------------------------ enums */
/* Gating of the router scores (the workloads' three families):
 *  SOFTMAX_RENORM:      choose top-k by logit; w = softmax over the chosen k   (Mixtral shape)
 *  SOFTMAX:             choose top-k by logit; w = softmax over all E           (Qwen1.5-MoE)
 *  SIGMOID_BIAS_RENORM: s = sigmoid(logit); choose top-k by s + sel_bias;
 *                       w = s / sum of the chosen s                            (DeepSeek-V3)
 * In every mode w is then multiplied by `scale`.  Selection order: larger score first, ties to
 * the lower expert id.  The chosen set is written in ascending expert id order. */
enum moe_gating {
  MOE_GATING_SOFTMAX_RENORM = 0,
  MOE_GATING_SOFTMAX = 1,
  MOE_GATING_SIGMOID_BIAS_RENORM = 2
};

/* Expert weight storage inside a bundle. */
enum moe_wdtype {
  MOE_W_BF16 = 0,      /* bf16 weights                                                   */
  MOE_W_INT4_G128 = 1, /* symmetric INT4 codes + one bf16 scale per 128 reduction elements */
  MOE_W_NVFP4 = 2      /* NVFP4: FP4 E2M1 codes, one FP8 E4M3 scale per 16 reduction
                          elements, one fp32 scale per matrix (gate, up, down)            */
};

/* ------------------------------------------------------------------ expert bundles
 * An expert bundle is the single unit that is stored, checksummed, cached and copied: one
 * contiguous byte block holding everything one SwiGLU expert needs -- weights and, for INT4,
 * their group scales -- so that weights can never arrive without their scales ("Running 35B
 * MoE Models on 8GB GPUs ...", section "Technical Insight").
 *
 * Layout.  Weights are stored as "weight rows": the gate/up section holds 2I rows of K = H
 * (rows 0..I-1 = columns of Wg, rows I..2I-1 = columns of Wu), the down section H rows of
 * K = I (row h = column h of Wd).  Rows are grouped into 128-row tiles stored tile after
 * tile, row-tile major then K-tile (each section starts on a 256-byte boundary):
 *   bf16: tiles of 128 rows x 64 k (16384 B).  Inside a tile, row r's 16-byte chunk c
 *         (elements k = 8c..8c+7 of the tile) is at byte r*128 + ((c ^ (r % 8)) * 16): the
 *         128-byte-swizzled K-major image the tensor cores read from shared memory, so a
 *         tile moves with one bulk copy.
 *   int4: tiles of 128 rows x 128 k (one scale group, 8448 B): 16-byte chunk (c, r) at
 *         (c*128 + r)*16 holds the 32 codes k = 32c..32c+31 of row r as four little-endian
 *         32-bit words of eight codes, sign-magnitude: code k = 8w + 2p + h of word w (pair
 *         p = 0..3, half h = 0/1) has its magnitude in bits (4 + 16h + 4p) mod 32 .. +2 and its
 *         sign in bit (15 + 16h + 4p) mod 32.  The word rotated right by 4p and masked with
 *         0x80708070 is pair p as two bf16 subnormals q * 2^-129, which one bf16 multiply by
 *         scale * 2^129 dequantises.  The codes are followed by the rows' bf16 group scales
 *         at 8192 + 2r.
 *   nvfp4: tiles of 128 rows x 128 k (9216 B): 16-byte chunk (c, r) at (c*128 + r)*16 holds
 *         the 32 FP4 codes k = 32c..32c+31 of row r as four little-endian 32-bit words of
 *         eight codes.  Code k = 8w + 2p + h of word w (pair p, half h) is a nibble
 *         (sign, e1, e0, m) whose bits sit so that pair p, moved to bits m: 6 + 16h,
 *         e0: 7 + 16h, e1: 8 + 16h, sign: 15 + 16h, is two bf16 numbers of value
 *         E2M1(code) * 2^-126.  Pairs 0, 1, 2 get there by rotating the word right by 0, 6
 *         and 12 and masking with 0x81C081C0; pair 3 by rotating right by 2 (e0, e1, sign;
 *         mask 0x81808180) and by 10 (m; mask 0x00400040).  A bf16 multiply by
 *         (block scale * 2^119) then gives E2M1 * scale * 2^-7 exactly (at most 6 significant
 *         bits).  The codes are followed by each row's 8 E4M3 block scales (k = 16b..16b+15
 *         of the tile) at 8192 + 8r + b.  The three fp32 matrix scales (gate, up, down)
 *         follow the down section at global_scale_offset.
 *   gate_up_scale_offset / down_scale_offset give the scale block of the section's first tile.
 * Constraints: H and I multiples of 128.  */
typedef struct moe_bundle_layout {
  size_t total_bytes;
  size_t gate_up_offset, down_offset;               /* weights or codes               */
  size_t gate_up_scale_offset, down_scale_offset;   /* INT4 / NVFP4, else 0           */
  size_t global_scale_offset;                       /* NVFP4: 3 fp32, else 0          */
} moe_bundle_layout;

/* Fills *out for an expert of hidden size H, intermediate size I and storage `wdtype`.
 * Returns MOE_ERR_INVALID_ARG unless H, I are positive multiples of 128. */
int moe_bundle_layout_of(int H, int I, int wdtype, moe_bundle_layout* out);
/* Size in bytes of one bundle (0 for invalid arguments). */
size_t moe_bundle_bytes(int H, int I, int wdtype);

/* Packs one expert from its logical host tensors into a host bundle `dst` of
 * moe_bundle_bytes() bytes (host memory, caller-owned; pinned or not).
 *  bf16: wg, wu: [H][I] uint16 bf16 bits; wd: [I][H]; scale arguments NULL.
 *  int4: wg, wu: [H][I] int8 codes in [-7,7]; wd: [I][H] int8 codes;
 *        sg, su: [H/128][I] bf16 bits (scale of group h/128, column i); sd: [I/128][H].
 * Host only, synchronous.  Returns MOE_ERR_INVALID_ARG on a code outside [-7, 7] or a scale
 * that is not finite with magnitude below 0.5 (codes times scales then stay below 3.5). */
int moe_pack_bundle(int H, int I, int wdtype, const void* wg, const void* wu, const void* wd,
                    const uint16_t* sg, const uint16_t* su, const uint16_t* sd, void* dst);

/* Packs one NVFP4 expert into a host bundle `dst` of moe_bundle_bytes(H, I, MOE_W_NVFP4)
 * bytes.  The weight is W[k][n] = E2M1(code) * E4M3(block scale) * matrix scale, the block
 * being 16 consecutive reduction elements k.
 *  wg, wu: [H][I] uint8 FP4 E2M1 codes (bit 3 sign, bits 2-1 exponent, bit 0 mantissa; values
 *          0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives); wd: [I][H].
 *  sg, su: [H/16][I] FP8 E4M3 block scales (bias 7, subnormals; block k/16, column n);
 *          sd: [I/16][H].
 *  gs:     [3] fp32 matrix scales of gate, up and down.
 * Host only, synchronous.  Returns MOE_ERR_INVALID_ARG on a code above 15, a block scale with
 * the sign bit set or the NaN pattern 0x7F, or a matrix scale that is not finite or has
 * magnitude 2^120 or more. */
int moe_pack_bundle_nvfp4(int H, int I, const uint8_t* wg, const uint8_t* wu, const uint8_t* wd,
                          const uint8_t* sg, const uint8_t* su, const uint8_t* sd,
                          const float* gs, void* dst);

/* FNV-1a 64-bit hash of `bytes` bytes of host memory (the checksum expert caches verify). */
uint64_t moe_checksum64(const void* data, size_t bytes);

/* ------------------------------------------------------------------ step 1-3: routing
 * moe_route_topk -- router logits, top-k gating and dispatch for T tokens.
 *
 *  x          device [T][H] bf16 activations
 *  w_r        device [H][E] fp32 router weight (row-major)
 *  logit_bias device [E] fp32 added to every token's logits, or NULL
 *  sel_bias   device [E] fp32 added to sigmoid scores for selection only, or NULL
 *             (SIGMOID_BIAS_RENORM only)
 *  w_gate     device [H] bf16 shared-expert gate vector, or NULL; when given,
 *             shared_gate[t] = sigmoid(x[t] . w_gate) is written to `shared_gate` (device [T] fp32)
 *  forced_ids device [T][k] int32 expert ids to use instead of the router's selection (each
 *             row k distinct ids in [0,E)), or NULL.  Weights are still the gating of the
 *             router logits at those ids.
 *  outputs (device): ids [T][k] int32 (ascending expert id within a token unless forced),
 *             w [T][k] fp32, counts [E] int32, offsets [E+1] int32 (exclusive scan of counts),
 *             pos [T][k] int32 (row of (t,j) in expert-contiguous order, stable in t),
 *             src [T*k] int32 (src[pos[t][j]] = t*k + j),
 *             logits [T][E] fp32 or NULL (the fp32 logits incl. logit_bias),
 *             tie_flags [T] int32 or NULL: 0 = the k-th/(k+1)-th selection gap exceeded the
 *             fp32 error margin; 1 = the experts near the boundary were re-scored (see
 *             below); 2 = as 1 and the re-scored gap was still below 1e-6 (a logged
 *             near-tie).
 *  ws         device scratch of moe_route_workspace_size(T, H, E, k) bytes.  Its first 4 bytes
 *             hold an error word, cleared at the start of every call: 0 = no error; non-zero =
 *             a bounded wait inside the tensor-core router (batches of T >= 256 tokens) ran out
 *             of time and the call's outputs are invalid.  Read it with moe_workspace_error.
 * Limits: 1 <= k <= min(E, 8), E <= 256, T >= 0 (T == 0 writes zero counts/offsets),
 * H a multiple of 8.  Exact selection: experts whose fp32 selection score lies within 1e-4 of
 * the k-th are re-scored on the GPU (the dot product x . W_r[:, e] in compensated fp32 -- each
 * product and each addition split error-free into a sum and its rounding error, error of
 * order H * 2^-48 * sum |x w| -- then the bias and the gating function in fp64), so the
 * chosen set equals that of exact arithmetic
 * (except ties closer than 1e-6, flagged 2) whenever the fp32 logits are within 1e-4 of the
 * exact ones.  That holds for activations and router weights of the workloads' magnitudes
 * (|x| ~ N(0, 1), W_r ~ N(0, 0.02), H <= 16384: observed fp32 error below 1e-5); inputs whose
 * products x[h] * W_r[h][e] are much larger can have fp32 logit errors above the margin, and
 * a choice near the boundary is then not guaranteed to be the exact one.
 * Defined by: "NovaLLM ...", "2. Why MoE Is a Natural Breakthrough Point" (the router picks a
 * handful of experts per token); the histogram, exclusive scan and stable rank that follow are
 * the standard counting-sort dispatch, which the pages do not spell out. */
size_t moe_route_workspace_size(int T, int H, int E, int k);
int moe_route_topk(const uint16_t* x, const float* w_r, const float* logit_bias,
                   const float* sel_bias, const uint16_t* w_gate, const int32_t* forced_ids,
                   int T, int H, int E, int k, int gating, float scale,
                   int32_t* ids, float* w, int32_t* counts, int32_t* offsets, int32_t* pos,
                   int32_t* src, float* logits, float* shared_gate, int32_t* tie_flags,
                   void* ws, size_t ws_bytes, void* stream);

/* moe_route_topk_static -- moe_route_topk without a workspace, for callers that cannot
 * allocate device memory.  The pages describe no counterpart; it exists for callers such as a
 * plug-in inside a host framework that owns all device memory and forbids allocations of its
 * own, or a latency-critical path where cudaMalloc / cudaFree (and the synchronisation they
 * can cause) are not acceptable.
 *
 * Arguments, outputs and results are those of moe_route_topk; the scratch is a fixed 8 MiB
 * array in the library's device memory (one per GPU that loads the library, held until the
 * process exits).  Returns MOE_ERR_CAPACITY when moe_route_workspace_size(T, H, E, k) exceeds
 * 8 MiB: batches of fewer than 256 tokens fit for E <= 256 and H <= 8192, while larger batches
 * route on the tensor cores, whose split router image needs 6*H*E' bytes (E' = E + 1 rounded up
 * to 128) plus 4*H*E (for example 23 MiB at H = 7168, E = 256).  Calls no
 * allocating routine.  The first call on a device looks up the array's device address once
 * (cudaGetSymbolAddress with that device current); make that first call before any stream
 * capture.  Every call on a device shares the one array and it keeps the previous call's
 * contents (the call clears what must start at zero itself): calls that can overlap on the
 * GPU -- on different streams, or from different host threads -- race and must be serialised
 * by the caller.  The cached address belongs to the device's primary context: do not use this
 * entry point across cudaDeviceReset.
 * Errors: as moe_route_topk; a timed-out wait of the tensor-core router (T >= 256) is reported
 * through the array's error word, read with moe_route_static_error. */
int moe_route_topk_static(const uint16_t* x, const float* w_r, const float* logit_bias,
                          const float* sel_bias, const uint16_t* w_gate, const int32_t* forced_ids,
                          int T, int H, int E, int k, int gating, float scale, int32_t* ids,
                          float* w, int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* src,
                          float* logits, float* shared_gate, int32_t* tie_flags, void* stream);
/* Reads the error word of moe_route_topk_static's fixed scratch on the current device into
 * *code (host) after waiting for `stream`: 0 = the last call on this device ran without error;
 * non-zero = a bounded wait of the tensor-core router ran out of time and that call's outputs
 * are invalid.  Blocking.  The same sharing rule applies: a call still running on another
 * stream can overwrite the word. */
int moe_route_static_error(int32_t* code, void* stream);

/* ------------------------------------------------------------------ step 4: permute
 * x_perm[p][:] = x[src[p] / k][:] for p in [0, T*k).
 *  x device [T][H] bf16, src device [T*k] int32, x_perm device [T*k][H] bf16.
 * H a multiple of 8.  The pages define no permutation step: it is the gather that puts each
 * expert's tokens next to each other so that every selected expert's weights are read once per
 * batch ("NovaLLM ...", "3. Optimization #1 -- Expert-Level Streaming" asks only that the
 * experts a batch hits be loaded and run). */
int moe_permute(const uint16_t* x, const int32_t* src, int T, int k, int H, uint16_t* x_perm,
                void* stream);

/* ------------------------------------------------------------------ step 5: expert FFN
 * moe_grouped_swiglu -- for every expert e with rows [offsets[e], offsets[e+1]) of x_perm:
 *   h = bf16( silu(x Wg_e) * (x Wu_e) ),  y_perm[rows] = bf16( h Wd_e ),
 * with fp32 accumulation (INT4: code x bf16 activation products, the group scale applied
 * in fp32 or folded into a bf16 dequantised weight; NVFP4: the exact bf16 product of code and
 * block scale times the activation, the matrix scale applied to the fp32 sum).
 *  x_perm   device [rows_total][H] bf16, rows_total = offsets[E]
 *  offsets  device [E+1] int32 (from moe_route_topk)
 *  bundles  HOST array [E] of device pointers to packed bundles (NULL allowed for experts
 *           that receive no rows); copied into the kernel parameters, so the array may be
 *           reused as soon as the call returns
 *  y_perm   device [rows_total][H] bf16
 *  max_rows an upper bound of offsets[E] (T*k), used to size the launch; an expert whose rows
 *           reach outside [0, max_rows) is clipped to it and error 8 is recorded in the
 *           workspace error word (moe_workspace_error)
 *  ws       device scratch of moe_grouped_swiglu_workspace_size(max_rows, E, H, I, wdtype)
 * Limits: E <= 256, H and I multiples of 128.
 * Defined by: "NovaLLM ...", "3. Optimization #1 -- Expert-Level Streaming" (only the experts
 * the batch selected are touched; each expert is the unit of storage and compute) and
 * "Running 35B MoE Models on 8GB GPUs ...", "Technical Insight" (INT4 / NVFP4 expert weights
 * travel with their scales in one bundle).  The SwiGLU form of an expert is that of the
 * Mixtral-, Qwen1.5-MoE- and DeepSeek-V3-shaped models the workloads follow. */
size_t moe_grouped_swiglu_workspace_size(int max_rows, int E, int H, int I, int wdtype);
int moe_grouped_swiglu(const uint16_t* x_perm, const int32_t* offsets,
                       const void* const* bundles, int E, int H, int I, int wdtype,
                       int max_rows, uint16_t* y_perm, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------ step 6: combine
 * out[t] = bf16( sum_{j<k} w[t][j] * y_perm[pos[t][j]] + g_t * shared[t] ), fp32 inside,
 * j in order 0..k-1, g_t = shared_gate[t] (1 when shared_gate is NULL; the shared term is
 * skipped when shared is NULL).  If `residual` is not NULL, out[t] = bf16(residual[t] +
 * that bf16 value) (the residual stream of a stacked model).  If `out_normed` (device [T][H]
 * bf16) is not NULL it also receives the next layer's input of a pre-norm stack,
 *   out_normed[t] = bf16( out[t] / sqrt(mean_h out[t][h]^2 + norm_eps) )
 * computed from the bf16 values of out[t] (sum of squares in fp32); H <= 32768 then.
 *  y_perm device [T*k][H] bf16; pos, w device [T][k]; shared, residual, out device [T][H].
 * The pages define no combine step: it is the gate-weighted sum that undoes the permutation,
 * the usual form of a top-k MoE layer's output. */
int moe_combine(const uint16_t* y_perm, const int32_t* pos, const float* w, int T, int k,
                int H, const uint16_t* shared, const float* shared_gate,
                const uint16_t* residual, uint16_t* out, uint16_t* out_normed, float norm_eps,
                void* stream);

/* ------------------------------------------------------------------ expert-slot cache
 * A fixed pool of VRAM slots, each holding one expert bundle, filled from pinned host
 * bundles by cudaMemcpyAsync on the cache's own copy stream under LRU eviction ("Running 35B
 * MoE Models on 8GB GPUs ...", section "Technical Insight"; "The Billion-Token Bottleneck",
 * sections "Tiered Memory" and "2. Async Weight Streaming").
 *
 * Policy (exactly reproducible): one LRU over keys (layer, expert).  A request processes its
 * distinct experts in ascending id order; a hit moves the key to most-recently-used; a miss
 * takes the lowest free slot, else evicts the least-recently-used key (never one this request
 * already touched).  Eviction drops the slot (the pinned host copy stays).  A request that
 * needs more distinct bundles than there are slots fails with MOE_ERR_CAPACITY and changes
 * nothing.
 *
 * Prefetch (lookahead: "NovaLLM ...", "3. Optimization #1 -- Expert-Level Streaming" reads the
 * next layer ahead while the current one computes; "The Billion-Token Bottleneck", "Predictive
 * Prefetching: Looking into the Future", copies predicted experts with cudaMemcpyAsync before
 * the model reaches their layer -- its predictor is a trained draft router, which is not part
 * of this library).  A prefetch request for a layer is processed exactly like a request (same
 * order, same LRU updates, same slot choice) but only copies: nothing computes on it.  Its
 * prediction is a caller-given expert mask or, by default, the set of experts the layer's
 * previous request used (the previous decode step's routing of that layer).  A later request
 * that hits a prefetched bundle waits for its copy. */
typedef struct moe_expert_cache moe_expert_cache;

typedef struct moe_host_bundle {
  const void* ptr;    /* host bundle (pinned memory for asynchronous copies)          */
  size_t bytes;       /* must equal the cache's slot_bytes                             */
  uint64_t checksum;  /* moe_checksum64 of the bundle, verified at creation            */
} moe_host_bundle;

typedef struct moe_expert_cache_config {
  size_t slot_bytes;        /* bytes of one bundle (moe_bundle_bytes)                  */
  size_t capacity_bytes;    /* VRAM budget: n_slots = capacity_bytes / slot_bytes       */
  int n_layers, n_experts;  /* key space                                               */
  const moe_host_bundle* bundles; /* host array [n_layers * n_experts], layer-major    */
  int timeout_ms;           /* deadline of every bounded host wait (<= 0: 10000 ms)     */
  int verify_checksums;     /* 1: hash every bundle at creation (MOE_ERR_CORRUPT)      */
  int device;               /* CUDA device ordinal of the slots                        */
  int time_copies;          /* 1: bracket every miss copy with timing events           */
  int prefetch_next_layer;  /* 1: moe_layer_forward on layer l ends by prefetching layer
                               (l + 1) mod n_layers with that layer's previous expert set */
  int device_lru;           /* 1: keep the LRU state on the GPU.  moe_layer_forward then
                               decides hits and misses in a kernel and copies the misses with
                               a copy kernel reading the host bundles over the host link (the
                               bundles must be pinned, mapped and 16-byte aligned): no host
                               round trip, the call is fully asynchronous and can be captured
                               in a CUDA graph.  Same policy and trace as the host LRU.  The
                               host-side request / wait / release / evict / prefetch calls
                               return MOE_ERR_UNSUPPORTED; trace, stats and sync synchronise
                               the device.  A layer that needs more bundles than slots records
                               error 20 in the workspace error word instead of returning
                               MOE_ERR_CAPACITY.                                        */
  int copy_kernel;          /* 1: the host LRU copies a request's misses with one kernel
                               that reads the host bundles through their device-visible
                               addresses (bundles pinned, mapped, 16-byte aligned, and
                               slot_bytes a multiple of 16; else MOE_ERR_INVALID_ARG at
                               creation) instead of one copy-engine cudaMemcpyAsync per
                               bundle.  Same slots, events and trace.  The device LRU always
                               copies this way.                                          */
} moe_expert_cache_config;

/* One trace record per distinct expert of every request (and prefetch request), in
 * processing order. */
typedef struct moe_cache_event {
  int64_t request;          /* running request number (requests and prefetches share it)   */
  int32_t layer, expert;
  int32_t miss;             /* 0 = hit, 1 = miss (a copy was issued)                       */
  int32_t victim_layer, victim_expert;  /* -1 when no key was evicted                  */
  int32_t slot;
  int32_t prefetch;         /* 1 = record of a prefetch request                            */
} moe_cache_event;

typedef struct moe_cache_stats {
  int64_t requests, hits, misses, evictions;  /* requests / hits / misses: demand requests */
  int64_t bytes_h2d;        /* every copied bundle (misses and prefetch fills) * slot_bytes */
  int32_t n_slots, resident;
  int64_t prefetch_requests, prefetch_fills;
  int64_t prefetch_used;    /* demand hits on a prefetched bundle, counted on its first use */
} moe_cache_stats;

/* Creates a cache: allocates n_slots slots in one device allocation, a non-blocking copy
 * stream and per-slot events, and (verify_checksums) hashes every host bundle.
 * Errors: MOE_ERR_INVALID_ARG; MOE_ERR_CORRUPT when a bundle's hash differs from its
 * checksum (the index of the first bad bundle goes to *bad_index when not NULL);
 * MOE_ERR_NO_MEMORY; MOE_ERR_CUDA.  Nothing is left allocated on failure. */
int moe_expert_cache_create(const moe_expert_cache_config* cfg, moe_expert_cache** out,
                            int64_t* bad_index);
int moe_expert_cache_destroy(moe_expert_cache* cache);

/* Makes every expert whose used_mask[e] != 0 resident for `layer`.  used_mask: HOST [E] bytes.
 * On return slot_ptrs[e] (HOST array [E], caller-owned) holds the device address of expert
 * e's bundle for every used e (NULL for unused e).  Misses are copied on the cache's copy
 * stream, each after the release that ended the reads of the slot's previous bundle
 * (write-after-read guard: the victim layer's last-use event, see moe_expert_cache_release).
 * The slots of a request stay held until its layer is released: a request or prefetch that
 * would have to evict a held slot returns MOE_ERR_CAPACITY and changes nothing, so call
 * moe_expert_cache_release for a layer before any later request that could evict its slots
 * (moe_layer_forward releases its layer itself).  If defer_waits == 0, stream `compute` is
 * made to wait for every copied bundle before any work enqueued on it after this call; if
 * defer_waits == 1 the caller adds those waits per expert with moe_expert_cache_wait_expert
 * (so work on hit experts can start while misses are in flight).  n_missed (nullable)
 * receives the number of misses.  Host-side and non-blocking. */
int moe_expert_cache_request(moe_expert_cache* cache, int layer, const uint8_t* used_mask,
                             void* compute, int defer_waits, const void** slot_ptrs,
                             int32_t* n_missed);
/* Prefetch request for `layer`: mask = HOST [E] bytes (experts to make resident), or NULL for
 * the experts of the layer's previous request (no-op when the layer has none yet).  Copies
 * are issued on the copy stream after the copies already issued; each waits for the previous
 * readers of its slot.  *n_filled (nullable) receives the number of copies.  Host-side and
 * non-blocking.  MOE_ERR_CAPACITY as for a request. */
int moe_expert_cache_prefetch(moe_expert_cache* cache, int layer, const uint8_t* mask,
                              int32_t* n_filled);
/* Makes stream `compute` wait until (layer, expert)'s bundle has arrived (no-op for a hit). */
int moe_expert_cache_wait_expert(moe_expert_cache* cache, int layer, int expert, void* compute);
/* Marks the end of `layer`'s use of its slots on stream `compute`: records the layer's
 * last-use event, which later copies into those slots wait for, and releases the slots held by
 * the layer's requests so that they can be evicted again. */
int moe_expert_cache_release(moe_expert_cache* cache, int layer, void* compute);
/* Drops (layer, expert) from the cache; no-op when not resident.  Waits (bounded, else
 * MOE_ERR_TIMEOUT) for the layer's last release.  MOE_ERR_INVALID_ARG when the bundle's slot
 * is held by a request whose layer has not been released yet. */
int moe_expert_cache_evict(moe_expert_cache* cache, int layer, int expert);
/* Copies up to `cap` trace records (oldest first, since creation or the last reset) into
 * `buf` (host); *n receives the number of records available. */
int moe_expert_cache_trace(const moe_expert_cache* cache, moe_cache_event* buf, size_t cap,
                           size_t* n);
int moe_expert_cache_reset_trace(moe_expert_cache* cache);
int moe_expert_cache_stats(const moe_expert_cache* cache, moe_cache_stats* out);
/* Bounded wait until every copy issued so far has completed (MOE_ERR_TIMEOUT on deadline). */
int moe_expert_cache_sync(moe_expert_cache* cache);
/* With time_copies: waits (bounded) for the timed copies issued since the last call, then
 * returns their summed copy-engine time in *ms and their count in *n (copy busy time, for
 * the achieved H2D bandwidth).  Without time_copies: *ms = 0, *n = 0. */
int moe_expert_cache_copy_time(moe_expert_cache* cache, double* ms, int64_t* n);

/* ------------------------------------------------------------------ whole layer */
typedef struct moe_layer {
  int H, E, k, I, Is;        /* Is = shared-expert intermediate size, 0 = none          */
  int gating;                /* enum moe_gating                                          */
  float scale;               /* routed weight multiplier                                 */
  int wdtype;                /* enum moe_wdtype of routed and shared bundles            */
  int layer_index;           /* cache key                                                */
  int shared_gate_sigmoid;   /* 1: shared term scaled by sigmoid(x . w_gate), 0: by 1   */
  const float* w_r;          /* device [H][E] fp32                                       */
  const float* logit_bias;   /* device [E] fp32 or NULL                                  */
  const float* sel_bias;     /* device [E] fp32 or NULL                                  */
  const uint16_t* w_gate;    /* device [H] bf16, required when shared_gate_sigmoid       */
  const void* shared_bundle; /* device bundle of the shared expert (H, Is), or NULL      */
  const void* const* bundles;/* HOST array [E] of device bundles (all resident), or NULL
                                when a cache is attached                                 */
  float norm_eps;            /* epsilon of the optional RMS-normalised output (out_normed) */
} moe_layer;

/* Number of phase events moe_layer_forward can record (see moe_layer_stats). */
#define MOE_N_PHASE_EVENTS 6

typedef struct moe_layer_stats {
  int32_t n_unique;          /* out: distinct experts used (cache path; 0 otherwise)      */
  int32_t n_missed;          /* out: cache misses (0 without a cache)                     */
  int32_t n_launches;        /* out: CUDA kernels this call launched                      */
  int32_t shared_merged;     /* out: 1 if the shared expert ran inside the routed GEMM
                                launches (phase [2] is then empty and phases [3] / [4]
                                include it), else 0                                      */
  int32_t fused_decode;      /* out: 1 if the whole layer ran as one fused decode launch
                                (phases [1]-[5] are then recorded together after it, so
                                phase [0]-[1] is the whole layer)                         */
  /* in: NULL, or a host array of MOE_N_PHASE_EVENTS cudaEvent_t handles created by the
   * caller; the call records them on `stream` at phase boundaries:
   *   [0] start  [1] routing + dispatch + gather done  [2] shared expert done
   *   [3] routed gate/up GEMM done (cache path: hit experts' FFN done)
   *   [4] routed down GEMM done (cache path: missed experts' FFN done)  [5] combine done */
  void* const* phase_events;
} moe_layer_stats;

/* Bytes of scratch moe_layer_forward needs for T tokens (the scratch must start on a 256-byte
 * boundary, as every device allocation does). */
size_t moe_layer_workspace_size(const moe_layer* L, int T);

/* The whole layer forward: out[T][H] (device bf16) from x[T][H] (device bf16).
 *  forced_ids device [T][k] or NULL (routing trace injection, see moe_route_topk)
 *  residual   device [T][H] bf16 or NULL (out = residual + layer output, see moe_combine)
 *  out_normed device [T][H] bf16 or NULL: out RMS-normalised with L->norm_eps (moe_combine),
 *             the next layer's input when layers are stacked with pre-normalisation
 *  cache      NULL: every bundle is resident (L->bundles); else bundles come from the cache:
 *             the call reads the layer's expert-use mask back to the host (one small
 *             device-to-host copy and a bounded wait), requests residency, and overlaps the
 *             miss copies with the shared expert and with the experts that hit.
 *  st         host, or NULL (in: phase_events; out: counters).
 *  ids_out, w_out  device [T][k] or NULL: copies of the routing decision.
 *  ws, ws_bytes    device scratch of moe_layer_workspace_size(L, T) bytes, 256-byte aligned
 *             (MOE_ERR_INVALID_ARG otherwise).
 * With cache == NULL the call is fully asynchronous.
 * Defined by: "NovaLLM ...", "2. Why MoE Is a Natural Breakthrough Point" and "3. Optimization
 * #1 -- Expert-Level Streaming" (route, then run only the selected experts, whose weights are
 * streamed in on demand and overlapped with compute); "Running 35B MoE Models on 8GB GPUs ...",
 * "Technical Insight" (the cache sits between the router's output and the experts' compute). */
int moe_layer_forward(const moe_layer* L, const uint16_t* x, int T, const int32_t* forced_ids,
                      const uint16_t* residual, uint16_t* out, uint16_t* out_normed,
                      moe_expert_cache* cache, moe_layer_stats* st, int32_t* ids_out,
                      float* w_out, void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */

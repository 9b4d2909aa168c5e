// Expert-slot cache with the LRU state on the GPU.
//
// The host-side cache (cache.cpp) needs the layer's expert-use mask on the host before it can
// decide hits and misses, so every layer pays a device-to-host round trip and the stack cannot
// be captured in a CUDA graph.  Here the same policy runs in a one-CTA kernel right after
// routing, and a copy kernel brings the missed bundles in from the pinned host store (read
// through its device-visible address over the host link): the layer forward is a plain stream
// of kernels.  Pages: "Running 35B MoE Models on 8GB GPUs: How vvllm-ms Caches Experts in
// System RAM", section "Technical Insight" (router output checked against resident bundles,
// LRU eviction); "The Billion-Token Bottleneck", section "2. Async Weight Streaming".
//
// Policy, identical to the host cache: one LRU over keys (layer, expert); a request takes its
// distinct experts in ascending order; a hit becomes most recently used; a miss takes the
// lowest free slot, else evicts the least recently used key this request has not touched.
// Recency is a clock incremented on every touch: the LRU key is the slot with the smallest
// clock, and keys touched by the current request have clocks above the request's start.
#include "cache.h"

#include <vector>

#include "common.cuh"
#include "route.cuh"

namespace moe {

namespace {

constexpr int kLruThreads = 256;
constexpr int kCopyCtas = 32, kCopyThreads = 512;
constexpr int64_t kTraceCap = int64_t(1) << 20;
constexpr int32_t kErrCapacity = 20;   // workspace error code: request larger than the cache

struct DevArgs {
  int64_t* ctl;
  int32_t* slot_key;
  int64_t* last_use;
  int32_t* key_slot;
  const void** ptrs;
  int32_t* lists;
  moe_cache_event* trace;
  int64_t trace_cap;
  char* slab;
  size_t slot_bytes;
  int n_slots, E;
};

// Block-wide argmin of (value, index) pairs; every thread gets the result.
__device__ void block_argmin(int64_t v, int i, int64_t* sv, int* si, int64_t& out_v, int& out_i) {
  const int tid = threadIdx.x;
  sv[tid] = v;
  si[tid] = i;
  __syncthreads();
  for (int o = kLruThreads / 2; o > 0; o >>= 1) {
    if (tid < o) {
      const int64_t v2 = sv[tid + o];
      const int i2 = si[tid + o];
      if (v2 < sv[tid] || (v2 == sv[tid] && i2 < si[tid])) {
        sv[tid] = v2;
        si[tid] = i2;
      }
    }
    __syncthreads();
  }
  out_v = sv[0];
  out_i = si[0];
  __syncthreads();
}

__global__ void __launch_bounds__(kLruThreads)
lru_request_kernel(DevArgs a, int layer, const int32_t* __restrict__ counts,
                   int32_t* __restrict__ err) {
  __shared__ int used[kMaxExperts];
  __shared__ int64_t sv[kLruThreads];
  __shared__ int si[kLruThreads];
  __shared__ int n_used;
  const int tid = threadIdx.x, E = a.E;
  int32_t* hit_list = a.lists;
  int32_t* n_hit = a.lists + E;
  int32_t* miss_list = a.lists + E + 1;
  int32_t* miss_slot = a.lists + 2 * E + 1;
  int32_t* n_miss = a.lists + 3 * E + 1;
  if (tid == 0) n_used = 0;
  __syncthreads();
  for (int e = tid; e < E; e += kLruThreads) {
    used[e] = counts[e] > 0;
    if (used[e]) atomicAdd(&n_used, 1);
    a.ptrs[e] = nullptr;
  }
  __syncthreads();
  if (n_used > a.n_slots) {
    // capacity error: nothing changes, no expert runs
    if (tid == 0) {
      *n_hit = 0;
      *n_miss = 0;
      atomicExch(err, kErrCapacity);
    }
    return;
  }
  const int64_t req = a.ctl[kReq];
  const int64_t start = a.ctl[kClock];   // clocks above this were touched by this request
  int64_t clock = start;
  int nh = 0, nm = 0;
  for (int e = 0; e < E; ++e) {
    if (!used[e]) continue;   // uniform across the block
    const int key = layer * E + e;
    int slot = a.key_slot[key];
    int vl = -1, ve = -1, miss = 0;
    if (slot < 0) {
      miss = 1;
      // lowest free slot
      int64_t best_v = INT64_MAX;
      int best_i = 0x7fffffff;
      for (int s = tid; s < a.n_slots; s += kLruThreads)
        if (a.slot_key[s] < 0 && s < best_i) best_i = s;
      int64_t fv;
      int fi;
      block_argmin(best_i == 0x7fffffff ? INT64_MAX : 0, best_i, sv, si, fv, fi);
      if (fv == 0) {
        slot = fi;
      } else {
        // least recently used slot not touched by this request
        best_v = INT64_MAX;
        best_i = 0x7fffffff;
        for (int s = tid; s < a.n_slots; s += kLruThreads) {
          const int64_t lu = a.last_use[s];
          if (lu <= start && (lu < best_v || (lu == best_v && s < best_i))) {
            best_v = lu;
            best_i = s;
          }
        }
        int64_t lv;
        block_argmin(best_v, best_i, sv, si, lv, slot);
        if (slot >= a.n_slots) {   // cannot happen while n_used <= n_slots; stop cleanly
          if (tid == 0) atomicExch(err, kErrCapacity);
          break;
        }
        const int victim = a.slot_key[slot];
        vl = victim / E;
        ve = victim % E;
        if (tid == 0) {
          a.key_slot[victim] = -1;
          a.ctl[kEvictions] += 1;
        }
      }
      if (tid == 0) {
        a.slot_key[slot] = key;
        a.key_slot[key] = slot;
        miss_list[nm] = e;
        miss_slot[nm] = slot;
        a.ctl[kMisses] += 1;
        a.ctl[kBytes] += (int64_t)a.slot_bytes;
      }
      ++nm;
    } else {
      if (tid == 0) {
        hit_list[nh] = e;
        a.ctl[kHits] += 1;
      }
      ++nh;
    }
    ++clock;
    if (tid == 0) {
      a.last_use[slot] = clock;
      a.ptrs[e] = a.slab + (size_t)slot * a.slot_bytes;
      const int64_t n = a.ctl[kTraceN];
      if (n < a.trace_cap) {
        moe_cache_event ev;
        ev.request = req;
        ev.layer = layer;
        ev.expert = e;
        ev.miss = miss;
        ev.victim_layer = vl;
        ev.victim_expert = ve;
        ev.slot = slot;
        ev.prefetch = 0;
        a.trace[n] = ev;
        a.ctl[kTraceN] = n + 1;
      } else {
        a.ctl[kOverflow] = 1;
      }
    }
    __syncthreads();   // the next expert's decisions see this one's table updates
  }
  if (tid == 0) {
    *n_hit = nh;
    *n_miss = nm;
    a.ctl[kClock] = clock;
    a.ctl[kReq] = req + 1;
  }
}

// One bundle from its device-visible host address into a slot: 16-byte loads over the host
// link, four in flight per thread, the grid striding through the bundle.
__device__ __forceinline__ void copy_bundle(const uint4* __restrict__ s, uint4* __restrict__ d,
                                            size_t n16) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 v0 = s[i], v1 = s[i + stride], v2 = s[i + 2 * stride], v3 = s[i + 3 * stride];
    d[i] = v0;
    d[i + stride] = v1;
    d[i + 2 * stride] = v2;
    d[i + 3 * stride] = v3;
  }
  for (; i < n16; i += stride) d[i] = s[i];
}

// Copies the missed bundles of the latest request from the host store into their slots.
__global__ void __launch_bounds__(kCopyThreads)
bundle_copy_kernel(DevArgs a, int layer, const void* const* __restrict__ src) {
  const int E = a.E;
  const int nm = a.lists[3 * E + 1];
  const int32_t* miss_list = a.lists + E + 1;
  const int32_t* miss_slot = a.lists + 2 * E + 1;
  const size_t n16 = a.slot_bytes / 16;
  for (int j = 0; j < nm; ++j)
    copy_bundle(static_cast<const uint4*>(src[(size_t)layer * E + miss_list[j]]),
                reinterpret_cast<uint4*>(a.slab + (size_t)miss_slot[j] * a.slot_bytes), n16);
}

// The fills of one host-LRU request: keys (layer * E + expert) and their slots, by value.
struct FillList {
  int n;
  int32_t key[kMaxExperts];
  int32_t slot[kMaxExperts];
};

__global__ void __launch_bounds__(kCopyThreads)
slot_fill_kernel(const void* const* __restrict__ src, char* __restrict__ slab, size_t slot_bytes,
                 FillList f) {
  const size_t n16 = slot_bytes / 16;
  for (int j = 0; j < f.n; ++j)
    copy_bundle(static_cast<const uint4*>(src[f.key[j]]),
                reinterpret_cast<uint4*>(slab + (size_t)f.slot[j] * slot_bytes), n16);
}

__global__ void init_kernel(int32_t* slot_key, int n_slots, int64_t* last_use, int32_t* key_slot,
                            int n_keys, int64_t* ctl) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n_slots) {
    slot_key[i] = -1;
    last_use[i] = 0;
  }
  if (i < n_keys) key_slot[i] = -1;
  if (i < kDevCtl) ctl[i] = 0;
}

DevArgs args_of(moe_expert_cache* c) {
  DevArgs a;
  a.ctl = c->d_ctl;
  a.slot_key = c->d_slot_key;
  a.last_use = c->d_last_use;
  a.key_slot = c->d_key_slot;
  a.ptrs = c->d_ptrs;
  a.lists = c->d_lists;
  a.trace = c->d_trace;
  a.trace_cap = c->trace_cap;
  a.slab = c->slab;
  a.slot_bytes = c->slot_bytes;
  a.n_slots = c->n_slots;
  a.E = c->E;
  return a;
}

}  // namespace

int cache_src_init(moe_expert_cache* c) {
  const size_t nk = (size_t)c->L * c->E;
  if (c->slot_bytes % 16) return MOE_ERR_INVALID_ARG;
  MOE_CUDA_TRY(cudaMalloc(&c->d_src, sizeof(void*) * nk));
  // device-visible addresses of the host bundles (pinned memory is mapped)
  std::vector<const void*> src(nk);
  for (size_t i = 0; i < nk; ++i) {
    void* dp = nullptr;
    const cudaError_t e = cudaHostGetDevicePointer(&dp, const_cast<void*>(c->bundles[i].ptr), 0);
    if (e != cudaSuccess || (reinterpret_cast<uintptr_t>(dp) & 15u)) {
      cudaGetLastError();
      return MOE_ERR_INVALID_ARG;   // not pinned (mapped) host memory, or not 16-byte aligned
    }
    src[i] = dp;
  }
  MOE_CUDA_TRY(cudaMemcpy(c->d_src, src.data(), sizeof(void*) * nk, cudaMemcpyHostToDevice));
  return MOE_OK;
}

int cache_dev_init(moe_expert_cache* c) {
  const size_t nk = (size_t)c->L * c->E;
  MOE_CUDA_TRY(cudaMalloc(&c->d_ctl, sizeof(int64_t) * kDevCtl));
  MOE_CUDA_TRY(cudaMalloc(&c->d_slot_key, sizeof(int32_t) * c->n_slots));
  MOE_CUDA_TRY(cudaMalloc(&c->d_last_use, sizeof(int64_t) * c->n_slots));
  MOE_CUDA_TRY(cudaMalloc(&c->d_key_slot, sizeof(int32_t) * nk));
  MOE_CUDA_TRY(cudaMalloc(&c->d_ptrs, sizeof(void*) * c->E));
  MOE_CUDA_TRY(cudaMalloc(&c->d_lists, sizeof(int32_t) * (3 * c->E + 2)));
  c->trace_cap = kTraceCap;
  MOE_CUDA_TRY(cudaMalloc(&c->d_trace, sizeof(moe_cache_event) * c->trace_cap));
  MOE_CUDA_TRY(cudaEventCreateWithFlags(&c->dev_lru_done, cudaEventDisableTiming));
  MOE_CUDA_TRY(cudaEventCreateWithFlags(&c->dev_copy_done, cudaEventDisableTiming));
  const int r = cache_src_init(c);
  if (r != MOE_OK) return r;
  const int n = (int)std::max<size_t>(std::max<size_t>(nk, c->n_slots), kDevCtl);
  init_kernel<<<ceil_div(n, 256), 256>>>(c->d_slot_key, c->n_slots, c->d_last_use,
                                         c->d_key_slot, (int)nk, c->d_ctl);
  MOE_LAUNCH_CHECK();
  MOE_CUDA_TRY(cudaDeviceSynchronize());
  return MOE_OK;
}

int cache_fill_slots(moe_expert_cache* c, int n, const int32_t* keys, const int32_t* slots) {
  if (n <= 0) return MOE_OK;
  if (n > kMaxExperts || !c->d_src) return MOE_ERR_INVALID_ARG;
  FillList f;
  f.n = n;
  for (int j = 0; j < n; ++j) {
    f.key[j] = keys[j];
    f.slot[j] = slots[j];
  }
  slot_fill_kernel<<<kCopyCtas, kCopyThreads, 0, c->copy>>>(c->d_src, c->slab, c->slot_bytes, f);
  MOE_COUNT_LAUNCH();
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

void cache_dev_free(moe_expert_cache* c) {
  if (c->dev_lru_done) cudaEventDestroy(c->dev_lru_done);
  if (c->dev_copy_done) cudaEventDestroy(c->dev_copy_done);
  c->dev_lru_done = c->dev_copy_done = nullptr;
  cudaFree(c->d_ctl);
  cudaFree(c->d_slot_key);
  cudaFree(c->d_last_use);
  cudaFree(c->d_key_slot);
  cudaFree(c->d_src);
  cudaFree(c->d_ptrs);
  cudaFree(c->d_lists);
  cudaFree(c->d_trace);
}

int cache_dev_request(moe_expert_cache* c, int layer, const int32_t* counts, cudaStream_t s0,
                      int32_t* err) {
  DevArgs a = args_of(c);
  lru_request_kernel<<<1, kLruThreads, 0, s0>>>(a, layer, counts, err);
  MOE_COUNT_LAUNCH();
  MOE_LAUNCH_CHECK();
  // the copies run on the copy stream beside the hit experts' compute; the victims are never
  // slots of this request, and every earlier reader of a slot ran before on s0
  MOE_CUDA_TRY(cudaEventRecord(c->dev_lru_done, s0));
  MOE_CUDA_TRY(cudaStreamWaitEvent(c->copy, c->dev_lru_done, 0));
  bundle_copy_kernel<<<kCopyCtas, kCopyThreads, 0, c->copy>>>(a, layer, c->d_src);
  MOE_COUNT_LAUNCH();
  MOE_LAUNCH_CHECK();
  MOE_CUDA_TRY(cudaEventRecord(c->dev_copy_done, c->copy));
  return MOE_OK;
}

int cache_dev_wait_copies(moe_expert_cache* c, cudaStream_t s0) {
  MOE_CUDA_TRY(cudaStreamWaitEvent(s0, c->dev_copy_done, 0));
  return MOE_OK;
}

}  // namespace moe

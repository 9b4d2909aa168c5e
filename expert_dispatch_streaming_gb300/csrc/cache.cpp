// Expert-slot cache: fixed VRAM slots filled on demand from pinned host bundles.
//
// Pages: "Running 35B MoE Models on 8GB GPUs: How vvllm-ms Caches Experts in System RAM",
// section "Technical Insight" (router output is intercepted before expert computation,
// residency of each expert bundle is checked, misses evict the least-recently-used bundles);
// "The Billion-Token Bottleneck", sections "Tiered Memory" (HBM hot tier over a host tier)
// and "2. Async Weight Streaming" (cudaMemcpyAsync of a missing expert's weights);
// "NovaLLM: Running Massive MoE Models Fully In-Memory", "Optimization #2" (every bundle stays
// resident in pinned host memory, so an evicted slot is simply dropped).
//
// A miss is copied by the copy engine (one cudaMemcpyAsync per bundle) or, with copy_kernel,
// by one kernel per request that reads the bundles through their device-visible host
// addresses (SM loads over the host link; on GB300's NVLink-C2C this held ~190 GB/s in every
// run, where the copy engine reached 190 GB/s in some runs and 90-140 GB/s in others).
//
// Ordering on the GPU, without any host wait in the steady state:
//  - a fill of slot s runs on the cache's copy stream after the event recorded when the
//    layer that last read s released it (write-after-read guard).  A slot whose reader has not
//    been released yet is never evicted: a request that would evict one is refused
//    (MOE_ERR_CAPACITY) before it changes anything, so the guard's event always exists;
//  - each fill records ready[s]; compute work that reads s waits on it (or on last_copy,
//    which follows every fill issued so far, since fills are serialised on one stream).
// Every host wait on the GPU is a polling loop with a deadline (MOE_ERR_TIMEOUT).
#include "cache.h"

#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <thread>
#include <vector>

#include "common.cuh"
#include "route.cuh"

namespace moe {

int cache_wait_event(moe_expert_cache* c, cudaEvent_t ev) {
  const auto t0 = std::chrono::steady_clock::now();
  for (long spin = 0;; ++spin) {
    const cudaError_t r = cudaEventQuery(ev);
    if (r == cudaSuccess) return MOE_OK;
    if (r != cudaErrorNotReady) return fail_cuda(r);
    if (std::chrono::steady_clock::now() - t0 > std::chrono::milliseconds(c->timeout_ms))
      return MOE_ERR_TIMEOUT;
    if (spin > 64) std::this_thread::yield();
  }
}

// time_copies: an event pair around each copy (or fill kernel) on the copy stream
static cudaError_t timed_copy_begin(moe_expert_cache* c) {
  if (!c->time_copies) return cudaSuccess;
  std::pair<cudaEvent_t, cudaEvent_t> tev{nullptr, nullptr};
  if (c->pool.empty()) {
    cudaError_t e = cudaEventCreate(&tev.first);
    if (e == cudaSuccess) e = cudaEventCreate(&tev.second);
    if (e != cudaSuccess) return e;
  } else {
    tev = c->pool.back();
    c->pool.pop_back();
  }
  c->timed.push_back(tev);
  return cudaEventRecord(tev.first, c->copy);
}
static cudaError_t timed_copy_end(moe_expert_cache* c) {
  if (!c->time_copies) return cudaSuccess;
  return cudaEventRecord(c->timed.back().second, c->copy);
}

static void destroy_all(moe_expert_cache* c) {
  if (!c) return;
  int cur = -1;
  cudaGetDevice(&cur);
  cudaSetDevice(c->device);
  if (c->copy) cudaStreamSynchronize(c->copy);
  cache_dev_free(c);   // device LRU state and the bundle address table (if any)
  for (auto e : c->ready) if (e) cudaEventDestroy(e);
  for (auto& pr : c->timed) { cudaEventDestroy(pr.first); cudaEventDestroy(pr.second); }
  for (auto& pr : c->pool) { cudaEventDestroy(pr.first); cudaEventDestroy(pr.second); }
  for (auto e : c->layer_done) if (e) cudaEventDestroy(e);
  if (c->last_copy) cudaEventDestroy(c->last_copy);
  if (c->d2h) cudaEventDestroy(c->d2h);
  if (c->copy) cudaStreamDestroy(c->copy);
  if (c->slab) cudaFree(c->slab);
  if (c->host_counts) cudaFreeHost(c->host_counts);
  if (cur >= 0) cudaSetDevice(cur);
  c->magic = 0;
  delete c;
}

static long long key_of(const moe_expert_cache* c, int layer, int e) {
  return (long long)layer * c->E + e;
}

// Picks the slot for a missing key: lowest free slot, else the LRU key not touched by this
// request (touched keys sit at the MRU end, so this is the LRU key).
static int take_slot(moe_expert_cache* c, long long req, int* vl, int* ve) {
  *vl = *ve = -1;
  if (!c->free_slots.empty()) {
    const int s = *c->free_slots.begin();
    c->free_slots.erase(c->free_slots.begin());
    return s;
  }
  for (auto it = c->order.begin(); it != c->order.end(); ++it) {
    const long long k = *it;
    const int s = c->where[k].first;
    if (c->slot_fill_req[s] == req) continue;  // (defensive) never a key of this request
    *vl = (int)(k / c->E);
    *ve = (int)(k % c->E);
    c->where.erase(k);
    c->order.erase(it);
    c->slot_key[s] = -1;
    c->st.evictions++;
    return s;
  }
  return -1;
}

// True when processing `used` for `layer` would evict a slot still held by a demand request
// that has not been released (its reads may still be in flight and no last-use event covers
// them).  The victims are the keys take_slot would pick: once the free slots are used up, the
// least-recently-used keys that are not hits of this request.
static bool evicts_held_slot(const moe_expert_cache* c, int layer, const uint8_t* used) {
  int n_miss = 0;
  std::vector<char> hit(c->E, 0);
  for (int e = 0; e < c->E; ++e) {
    if (!used[e]) continue;
    if (c->where.count(key_of(c, layer, e))) hit[e] = 1;
    else ++n_miss;
  }
  int victims = n_miss - (int)c->free_slots.size();
  for (auto it = c->order.begin(); victims > 0 && it != c->order.end(); ++it) {
    const long long k = *it;
    if (k / c->E == layer && hit[k % c->E]) continue;
    if (c->slot_holder[c->where.at(k).first] >= 0) return true;
    --victims;
  }
  return false;
}

// Host function of the delay hook: holds the copy stream for the given milliseconds.
static void CUDART_CB sleep_on_stream(void* ms) {
  std::this_thread::sleep_for(std::chrono::milliseconds((long)(intptr_t)ms));
}

// Drops `key` from slot `slot` (the slot becomes free); used when its fill could not be issued.
static void drop_key(moe_expert_cache* c, long long key, int slot) {
  auto f = c->where.find(key);
  if (f != c->where.end()) {
    c->order.erase(f->second.second);
    c->where.erase(f);
  }
  c->slot_key[slot] = -1;
  c->slot_pending[slot] = 0;
  c->slot_prefetched[slot] = 0;
  c->slot_holder[slot] = -1;
  c->free_slots.insert(slot);
}

// One request over the distinct experts of `used` (ascending): the LRU update, slot choice and
// miss copies shared by demand requests and prefetch requests.
//
// A miss whose copy cannot be issued ends the request with MOE_ERR_CUDA: its trace record (the
// policy's decision, victim included) is kept, the key is then dropped again (its slot is
// free, as after an explicit eviction), the experts after it are not processed, and the copies
// of the misses before it are issued as usual.  The trace therefore stays that of the LRU
// policy applied to the processed prefix followed by an eviction of the failed key.
static int process(moe_expert_cache* c, int layer, const uint8_t* used, bool prefetch,
                   const void** slot_ptrs, std::vector<int>* hits, std::vector<int>* misses,
                   std::vector<int>* wait_slots) {
  if (!c || !used || layer < 0 || layer >= c->L) return MOE_ERR_INVALID_ARG;
  int n_used = 0;
  for (int e = 0; e < c->E; ++e) n_used += used[e] != 0;
  if (n_used > c->n_slots) return MOE_ERR_CAPACITY;
  if (evicts_held_slot(c, layer, used)) return MOE_ERR_CAPACITY;
  const long long req = c->req++;
  if (prefetch) c->st.prefetch_requests++;
  else c->st.requests++;
  std::vector<int>& ls = c->layer_slots[layer];
  if (!prefetch) {
    ls.clear();
    c->layer_last[layer].clear();
  }
  std::vector<char> touched_slot(c->n_slots, 0);
  bool any_miss = false;
  int status = MOE_OK;
  std::vector<int32_t> fill_key, fill_slot;   // copy_kernel: this request's fills
  for (int e = 0; e < c->E; ++e) {
    if (slot_ptrs) slot_ptrs[e] = nullptr;
    if (!used[e]) continue;
    const long long k = key_of(c, layer, e);
    moe_cache_event ev{};
    ev.request = req;
    ev.layer = layer;
    ev.expert = e;
    ev.victim_layer = ev.victim_expert = -1;
    ev.prefetch = prefetch ? 1 : 0;
    int slot;
    auto f = c->where.find(k);
    if (f != c->where.end()) {
      slot = f->second.first;
      c->order.erase(f->second.second);
      c->order.push_back(k);
      f->second.second = std::prev(c->order.end());
      ev.miss = 0;
      if (!prefetch) {
        c->st.hits++;
        if (c->slot_prefetched[slot]) {
          c->st.prefetch_used++;
          c->slot_prefetched[slot] = 0;
        }
        if (c->slot_pending[slot] && wait_slots) wait_slots->push_back(slot);
        if (hits) hits->push_back(e);
      }
    } else {
      int vl, ve;
      slot = take_slot(c, req, &vl, &ve);
      if (slot < 0 || touched_slot[slot]) return MOE_ERR_CAPACITY;
      c->order.push_back(k);
      c->where[k] = {slot, std::prev(c->order.end())};
      c->slot_key[slot] = k;
      c->slot_fill_req[slot] = req;
      ev.miss = 1;
      ev.victim_layer = vl;
      ev.victim_expert = ve;
      if (prefetch) c->st.prefetch_fills++;
      else c->st.misses++;
      // write-after-read guard: the victim's layer must have finished reading this slot
      if (vl >= 0 && c->layer_done_valid[vl])
        MOE_CUDA_TRY(cudaStreamWaitEvent(c->copy, c->layer_done[vl], 0));
      const long long nth = ++c->fault_misses;
      if (nth == c->fault_delay_at)
        MOE_CUDA_TRY(cudaLaunchHostFunc(c->copy, sleep_on_stream,
                                        (void*)(intptr_t)c->fault_delay_ms));
      cudaError_t ce = nth == c->fault_fail_at ? cudaErrorUnknown : cudaSuccess;
      if (ce == cudaSuccess) {
        if (c->copy_kernel) {
          fill_key.push_back((int32_t)((size_t)layer * c->E + e));   // copied after the loop
          fill_slot.push_back(slot);
        } else {
          const moe_host_bundle& hb = c->bundles[(size_t)layer * c->E + e];
          ce = timed_copy_begin(c);
          if (ce == cudaSuccess) {
            ce = cudaMemcpyAsync(c->slab + (size_t)slot * c->slot_bytes, hb.ptr, hb.bytes,
                                 cudaMemcpyHostToDevice, c->copy);
            if (ce == cudaSuccess) ce = timed_copy_end(c);
            if (ce != cudaSuccess && c->time_copies) {   // the timing pair never completed
              c->pool.push_back(c->timed.back());
              c->timed.pop_back();
            }
          }
          if (ce == cudaSuccess) ce = cudaEventRecord(c->ready[slot], c->copy);
        }
      }
      if (ce != cudaSuccess) {
        // the decision stands in the trace; the key does not stay resident without its bytes
        ev.slot = slot;
        c->trace.push_back(ev);
        if (!prefetch) c->layer_last[layer].push_back(e);
        drop_key(c, k, slot);
        status = fail_cuda(ce);
        break;
      }
      c->st.bytes_h2d += (int64_t)c->slot_bytes;
      c->slot_pending[slot] = prefetch ? 1 : 0;   // a demand miss is waited for via last_copy
      c->slot_prefetched[slot] = prefetch ? 1 : 0;
      any_miss = true;
      if (misses) misses->push_back(e);
    }
    touched_slot[slot] = 1;
    ev.slot = slot;
    if (!prefetch) {
      ls.push_back(slot);
      c->layer_last[layer].push_back(e);
      c->slot_holder[slot] = layer;   // until the layer is released
    }
    c->trace.push_back(ev);
    if (slot_ptrs) slot_ptrs[e] = c->slab + (size_t)slot * c->slot_bytes;
  }
  if (!fill_key.empty()) {
    // one kernel for all fills, after every victim's write-after-read guard above
    MOE_CUDA_TRY(timed_copy_begin(c));
    const int r = cache_fill_slots(c, (int)fill_key.size(), fill_key.data(), fill_slot.data());
    if (r != MOE_OK) {
      if (c->time_copies) {   // the pair's end was never recorded: back to the pool
        c->pool.push_back(c->timed.back());
        c->timed.pop_back();
      }
      return r;
    }
    MOE_CUDA_TRY(timed_copy_end(c));
    for (int32_t sl : fill_slot) MOE_CUDA_TRY(cudaEventRecord(c->ready[sl], c->copy));
  }
  if (any_miss) MOE_CUDA_TRY(cudaEventRecord(c->last_copy, c->copy));
  c->st.resident = (int32_t)c->where.size();
  return status;
}

int cache_request_split(moe_expert_cache* c, int layer, const uint8_t* used, cudaStream_t compute,
                        const void** slot_ptrs, std::vector<int>* hits,
                        std::vector<int>* misses, std::vector<int>* wait_slots) {
  (void)compute;
  return process(c, layer, used, false, slot_ptrs, hits, misses, wait_slots);
}

int cache_release(moe_expert_cache* c, int layer, cudaStream_t compute) {
  MOE_CUDA_TRY(cudaEventRecord(c->layer_done[layer], compute));
  c->layer_done_valid[layer] = 1;
  for (int& h : c->slot_holder)
    if (h == layer) h = -1;
  return MOE_OK;
}

int cache_prefetch(moe_expert_cache* c, int layer, const uint8_t* mask, int32_t* n_filled) {
  if (n_filled) *n_filled = 0;
  if (!c || layer < 0 || layer >= c->L) return MOE_ERR_INVALID_ARG;
  std::vector<uint8_t> m(c->E, 0);
  if (mask) {
    for (int e = 0; e < c->E; ++e) m[e] = mask[e] != 0;
  } else {
    if (c->layer_last[layer].empty()) return MOE_OK;   // nothing to predict from yet
    for (int e : c->layer_last[layer]) m[e] = 1;
  }
  std::vector<int> fills;
  const int r = process(c, layer, m.data(), true, nullptr, nullptr, &fills, nullptr);
  if (r == MOE_OK && n_filled) *n_filled = (int32_t)fills.size();
  return r;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_expert_cache_create(const moe_expert_cache_config* cfg, moe_expert_cache** out,
                            int64_t* bad_index) {
  if (bad_index) *bad_index = -1;
  if (!cfg || !out || cfg->slot_bytes == 0 || cfg->n_layers <= 0 || cfg->n_experts <= 0 ||
      cfg->n_experts > kMaxExperts || !cfg->bundles)
    return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  const size_t nb = (size_t)cfg->n_layers * cfg->n_experts;
  for (size_t i = 0; i < nb; ++i)
    if (!cfg->bundles[i].ptr || cfg->bundles[i].bytes != cfg->slot_bytes)
      return MOE_ERR_INVALID_ARG;
  const size_t n_slots = cfg->capacity_bytes / cfg->slot_bytes;
  if (n_slots == 0 || n_slots > (1u << 30)) return MOE_ERR_INVALID_ARG;

  if (cfg->verify_checksums) {
    // bundles are hashed in parallel; each hash is the sequential FNV-1a of one bundle
    std::vector<char> bad(nb, 0);
    const unsigned nt = std::max(1u, std::min(32u, std::thread::hardware_concurrency()));
    std::vector<std::thread> th;
    for (unsigned w = 0; w < nt; ++w)
      th.emplace_back([&, w] {
        for (size_t i = w; i < nb; i += nt)
          bad[i] = moe_checksum64(cfg->bundles[i].ptr, cfg->bundles[i].bytes) !=
                   cfg->bundles[i].checksum;
      });
    for (auto& t : th) t.join();
    for (size_t i = 0; i < nb; ++i)
      if (bad[i]) {
        if (bad_index) *bad_index = (int64_t)i;
        return MOE_ERR_CORRUPT;
      }
  }

  auto* c = new moe_expert_cache();
  c->device = cfg->device;
  c->slot_bytes = cfg->slot_bytes;
  c->n_slots = (int)n_slots;
  c->L = cfg->n_layers;
  c->E = cfg->n_experts;
  c->timeout_ms = cfg->timeout_ms > 0 ? cfg->timeout_ms : 10000;
  c->time_copies = cfg->time_copies;
  c->bundles.assign(cfg->bundles, cfg->bundles + nb);
  int cur = -1;
  cudaGetDevice(&cur);
  cudaError_t err = cudaSetDevice(c->device);
  int status = MOE_OK;
  auto check = [&](cudaError_t e) {
    if (e != cudaSuccess && status == MOE_OK) {
      status = (e == cudaErrorMemoryAllocation) ? MOE_ERR_NO_MEMORY : fail_cuda(e);
      cudaGetLastError();
    }
  };
  check(err);
  if (status == MOE_OK) check(cudaMalloc(&c->slab, n_slots * cfg->slot_bytes));
  if (status == MOE_OK) check(cudaStreamCreateWithFlags(&c->copy, cudaStreamNonBlocking));
  if (status == MOE_OK) check(cudaMallocHost(&c->host_counts, sizeof(int32_t) * kMaxExperts));
  c->ready.assign(n_slots, nullptr);
  c->layer_done.assign(c->L, nullptr);
  for (size_t s = 0; s < n_slots && status == MOE_OK; ++s)
    check(cudaEventCreateWithFlags(&c->ready[s], cudaEventDisableTiming));
  for (int l = 0; l < c->L && status == MOE_OK; ++l)
    check(cudaEventCreateWithFlags(&c->layer_done[l], cudaEventDisableTiming));
  if (status == MOE_OK) check(cudaEventCreateWithFlags(&c->last_copy, cudaEventDisableTiming));
  if (status == MOE_OK) check(cudaEventCreateWithFlags(&c->d2h, cudaEventDisableTiming));
  if (cur >= 0) cudaSetDevice(cur);
  if (status != MOE_OK) {
    destroy_all(c);
    return status;
  }
  c->layer_done_valid.assign(c->L, 0);
  for (int s = 0; s < c->n_slots; ++s) c->free_slots.insert(s);
  c->slot_key.assign(n_slots, -1);
  c->slot_fill_req.assign(n_slots, -1);
  c->layer_slots.assign(c->L, {});
  c->layer_last.assign(c->L, {});
  c->slot_holder.assign(n_slots, -1);
  c->slot_pending.assign(n_slots, 0);
  c->slot_prefetched.assign(n_slots, 0);
  c->prefetch_next = cfg->prefetch_next_layer;
  // failure-test hooks (host LRU only): MOE_TEST_FAIL_COPY=n fails the n-th miss copy,
  // MOE_TEST_DELAY_COPY=n:ms holds the copy stream for ms milliseconds before the n-th
  if (const char* f = std::getenv("MOE_TEST_FAIL_COPY")) c->fault_fail_at = std::atoll(f);
  if (const char* d = std::getenv("MOE_TEST_DELAY_COPY")) {
    long long n = 0;
    int ms = 0;
    if (std::sscanf(d, "%lld:%d", &n, &ms) == 2 && n > 0 && ms > 0) {
      c->fault_delay_at = n;
      c->fault_delay_ms = ms;
    }
  }
  c->st.n_slots = c->n_slots;
  if (cfg->device_lru || cfg->copy_kernel) {
    c->device_lru = cfg->device_lru ? 1 : 0;
    c->copy_kernel = cfg->copy_kernel ? 1 : 0;
    cur = -1;
    cudaGetDevice(&cur);
    cudaSetDevice(c->device);
    const int r = c->device_lru ? cache_dev_init(c) : cache_src_init(c);
    if (cur >= 0) cudaSetDevice(cur);
    if (r != MOE_OK) {
      destroy_all(c);
      return r;
    }
  }
  c->magic = kCacheMagic;
  *out = c;
  return MOE_OK;
}

int moe_expert_cache_destroy(moe_expert_cache* cache) {
  if (!cache_live(cache)) return MOE_ERR_INVALID_ARG;
  destroy_all(cache);
  return MOE_OK;
}

int moe_expert_cache_request(moe_expert_cache* cache, int layer, const uint8_t* used_mask,
                             void* compute, int defer_waits, const void** slot_ptrs,
                             int32_t* n_missed) {
  if (!cache_live(cache)) return MOE_ERR_INVALID_ARG;
  if (cache->device_lru) return MOE_ERR_UNSUPPORTED;
  std::vector<int> misses, waits;
  const int r = cache_request_split(cache, layer, used_mask, (cudaStream_t)compute, slot_ptrs,
                                    nullptr, &misses, &waits);
  if (r != MOE_OK) return r;
  if (n_missed) *n_missed = (int32_t)misses.size();
  if (!defer_waits) {
    if (!misses.empty())
      MOE_CUDA_TRY(cudaStreamWaitEvent((cudaStream_t)compute, cache->last_copy, 0));
    for (int s : waits) {
      MOE_CUDA_TRY(cudaStreamWaitEvent((cudaStream_t)compute, cache->ready[s], 0));
      cache->slot_pending[s] = 0;
    }
  }
  return MOE_OK;
}

int moe_expert_cache_prefetch(moe_expert_cache* cache, int layer, const uint8_t* mask,
                              int32_t* n_filled) {
  if (!cache_live(cache)) return MOE_ERR_INVALID_ARG;
  if (cache->device_lru) return MOE_ERR_UNSUPPORTED;
  return cache_prefetch(cache, layer, mask, n_filled);
}

int moe_expert_cache_wait_expert(moe_expert_cache* cache, int layer, int expert,
                                 void* compute) {
  if (!cache_live(cache) || layer < 0 || layer >= cache->L || expert < 0 || expert >= cache->E)
    return MOE_ERR_INVALID_ARG;
  if (cache->device_lru) return MOE_ERR_UNSUPPORTED;
  auto f = cache->where.find(key_of(cache, layer, expert));
  if (f == cache->where.end()) return MOE_ERR_INVALID_ARG;
  const int slot = f->second.first;
  // filled by the latest request, or by a prefetch nothing has waited for yet
  if (cache->slot_fill_req[slot] == cache->req - 1 || cache->slot_pending[slot]) {
    MOE_CUDA_TRY(cudaStreamWaitEvent((cudaStream_t)compute, cache->ready[slot], 0));
    cache->slot_pending[slot] = 0;
  }
  return MOE_OK;
}

int moe_expert_cache_release(moe_expert_cache* cache, int layer, void* compute) {
  if (!cache_live(cache) || layer < 0 || layer >= cache->L) return MOE_ERR_INVALID_ARG;
  if (cache->device_lru) return MOE_ERR_UNSUPPORTED;
  return cache_release(cache, layer, (cudaStream_t)compute);
}

int moe_expert_cache_evict(moe_expert_cache* cache, int layer, int expert) {
  if (!cache_live(cache) || layer < 0 || layer >= cache->L || expert < 0 || expert >= cache->E)
    return MOE_ERR_INVALID_ARG;
  if (cache->device_lru) return MOE_ERR_UNSUPPORTED;
  auto f = cache->where.find(key_of(cache, layer, expert));
  if (f == cache->where.end()) return MOE_OK;
  const int slot = f->second.first;
  // a slot read by a request that has not been released: its reads may still be enqueued
  if (cache->slot_holder[slot] >= 0) return MOE_ERR_INVALID_ARG;
  if (cache->layer_done_valid[layer]) {
    const int r = cache_wait_event(cache, cache->layer_done[layer]);
    if (r != MOE_OK) return r;
  }
  cache->order.erase(f->second.second);
  cache->where.erase(f);
  cache->slot_key[slot] = -1;
  cache->slot_prefetched[slot] = 0;
  cache->free_slots.insert(slot);
  cache->st.evictions++;
  cache->st.resident = (int32_t)cache->where.size();
  return MOE_OK;
}

// Device-side LRU: copy its counters into the host stats / the trace into the host vector.
static int dev_sync_state(moe_expert_cache* c) {
  int64_t ctl[kDevCtl];
  MOE_CUDA_TRY(cudaDeviceSynchronize());
  MOE_CUDA_TRY(cudaMemcpy(ctl, c->d_ctl, sizeof(ctl), cudaMemcpyDeviceToHost));
  c->st.requests = ctl[kReq];
  c->st.hits = ctl[kHits];
  c->st.misses = ctl[kMisses];
  c->st.evictions = ctl[kEvictions];
  c->st.bytes_h2d = ctl[kBytes];
  const int64_t n = std::min(ctl[kTraceN], c->trace_cap);
  c->trace.resize((size_t)n);
  if (n > 0)
    MOE_CUDA_TRY(cudaMemcpy(c->trace.data(), c->d_trace, sizeof(moe_cache_event) * n,
                            cudaMemcpyDeviceToHost));
  std::vector<int32_t> sk(c->n_slots);
  MOE_CUDA_TRY(cudaMemcpy(sk.data(), c->d_slot_key, sizeof(int32_t) * c->n_slots,
                          cudaMemcpyDeviceToHost));
  int res = 0;
  for (int32_t k : sk) res += k >= 0;
  c->st.resident = res;
  return MOE_OK;
}

int moe_expert_cache_trace(const moe_expert_cache* cache, moe_cache_event* buf, size_t cap,
                           size_t* n) {
  if (!cache_live(cache) || !n) return MOE_ERR_INVALID_ARG;
  if (cache->device_lru) {
    const int r = dev_sync_state(const_cast<moe_expert_cache*>(cache));
    if (r != MOE_OK) return r;
  }
  *n = cache->trace.size();
  if (buf) std::memcpy(buf, cache->trace.data(), sizeof(moe_cache_event) * std::min(cap, *n));
  return MOE_OK;
}

int moe_expert_cache_reset_trace(moe_expert_cache* cache) {
  if (!cache_live(cache)) return MOE_ERR_INVALID_ARG;
  if (cache->device_lru) {
    MOE_CUDA_TRY(cudaDeviceSynchronize());
    MOE_CUDA_TRY(cudaMemset(cache->d_ctl + kTraceN, 0, sizeof(int64_t)));
  }
  cache->trace.clear();
  return MOE_OK;
}

int moe_expert_cache_stats(const moe_expert_cache* cache, moe_cache_stats* out) {
  if (!cache_live(cache) || !out) return MOE_ERR_INVALID_ARG;
  if (cache->device_lru) {
    const int r = dev_sync_state(const_cast<moe_expert_cache*>(cache));
    if (r != MOE_OK) return r;
  }
  *out = cache->st;
  return MOE_OK;
}

int moe_expert_cache_sync(moe_expert_cache* cache) {
  if (!cache_live(cache)) return MOE_ERR_INVALID_ARG;
  MOE_CUDA_TRY(cudaEventRecord(cache->last_copy, cache->copy));
  return cache_wait_event(cache, cache->last_copy);
}

int moe_expert_cache_copy_time(moe_expert_cache* cache, double* ms, int64_t* n) {
  if (!cache_live(cache) || !ms || !n) return MOE_ERR_INVALID_ARG;
  *ms = 0.0;
  *n = 0;
  for (auto& pr : cache->timed) {
    const int r = cache_wait_event(cache, pr.second);
    if (r != MOE_OK) return r;
    float t = 0.f;
    MOE_CUDA_TRY(cudaEventElapsedTime(&t, pr.first, pr.second));
    *ms += t;
    ++*n;
    cache->pool.push_back(pr);
  }
  cache->timed.clear();
  return MOE_OK;
}

}  // extern "C"

// Expert-slot cache internals shared by cache.cpp and the layer forward (internal).
#pragma once
#include <cuda_runtime.h>

#include <list>
#include <set>
#include <unordered_map>
#include <vector>

#include "../../include/moe.h"

// Set by moe_expert_cache_create and cleared just before the object is freed, so that a call
// on a destroyed cache is refused (best effort: the freed memory may have been reused).
constexpr uint32_t kCacheMagic = 0x43454F4Du;

struct moe_expert_cache {
  uint32_t magic = 0;
  int device = 0;
  size_t slot_bytes = 0;
  int n_slots = 0, L = 0, E = 0;
  int timeout_ms = 10000;
  std::vector<moe_host_bundle> bundles;
  char* slab = nullptr;                  // device, n_slots * slot_bytes
  cudaStream_t copy = nullptr;           // non-blocking copy stream
  std::vector<cudaEvent_t> ready;        // per slot: its last fill has landed
  std::vector<cudaEvent_t> layer_done;   // per layer: last release (end of reads)
  std::vector<char> layer_done_valid;
  cudaEvent_t last_copy = nullptr;       // after the most recent fill
  cudaEvent_t d2h = nullptr;             // routing read-back of the layer forward
  int32_t* host_counts = nullptr;        // pinned, [E]
  // LRU state
  std::list<long long> order;            // keys, LRU first
  std::unordered_map<long long, std::pair<int, std::list<long long>::iterator>> where;
  std::set<int> free_slots;
  std::vector<long long> slot_key;       // -1 = free
  std::vector<long long> slot_fill_req;  // request number of the slot's last fill
  std::vector<std::vector<int>> layer_slots;  // slots the layer's last request used
  std::vector<std::vector<int>> layer_last;   // experts of the layer's last (demand) request
  std::vector<int> slot_holder;          // layer whose demand request reads the slot and has
                                         // not been released yet, -1 = none
  std::vector<char> slot_pending;        // filled, and no compute has waited for it yet
  std::vector<char> slot_prefetched;     // filled by a prefetch, not yet used by a request
  int prefetch_next = 0;
  int copy_kernel = 0;                   // host LRU: misses copied by slot_fill_kernel
  // host-side fault hooks for failure tests (0 = off; set at creation from the environment):
  // the fault_fail_at-th miss copy of this cache fails as if its copy could not be issued, and
  // the fault_delay_at-th is preceded on the copy stream by a host function sleeping
  // fault_delay_ms
  long long fault_misses = 0, fault_fail_at = 0, fault_delay_at = 0;
  int fault_delay_ms = 0;
  std::vector<moe_cache_event> trace;
  moe_cache_stats st{};
  long long req = 0;
  // copy timing (time_copies): event pairs of copies not yet collected, and a free pool
  int time_copies = 0;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> timed, pool;
  // device-side LRU (device_lru): the policy state lives on the GPU and the layer forward
  // needs no host round trip (see cache_dev.cu)
  int device_lru = 0;
  int64_t* d_ctl = nullptr;         // [kDevCtl] counters (DevCtl indices)
  int32_t* d_slot_key = nullptr;    // [n_slots] key of the slot, -1 free
  int64_t* d_last_use = nullptr;    // [n_slots] clock of the slot's last touch
  int32_t* d_key_slot = nullptr;    // [L*E] slot of the key, -1 not resident
  const void** d_src = nullptr;     // [L*E] device-visible address of each host bundle
  const void** d_ptrs = nullptr;    // [E] bundle pointer table of the latest request
  int32_t* d_lists = nullptr;       // hit list [E], n_hit, miss list [E], miss slots [E], n_miss
  moe_cache_event* d_trace = nullptr;
  int64_t trace_cap = 0;
  cudaEvent_t dev_lru_done = nullptr, dev_copy_done = nullptr;
};

namespace moe {
inline bool cache_live(const moe_expert_cache* c) { return c && c->magic == kCacheMagic; }
int cache_wait_event(moe_expert_cache* c, cudaEvent_t ev);
// Request with the hit/miss split reported (used by the layer forward).  wait_slots (nullable)
// receives the slots of hits whose copy (a prefetch) no compute has waited for yet; the caller
// makes its compute stream wait on their ready events before using them.
int cache_request_split(moe_expert_cache* c, int layer, const uint8_t* used, cudaStream_t compute,
                        const void** slot_ptrs, std::vector<int>* hits, std::vector<int>* misses,
                        std::vector<int>* wait_slots = nullptr);
// Prefetch request (see moe_expert_cache_prefetch); mask NULL = the layer's last expert set.
int cache_prefetch(moe_expert_cache* c, int layer, const uint8_t* mask, int32_t* n_filled);
// End of `layer`'s reads of its slots on stream `compute`: records the layer's last-use event
// (later fills of those slots wait for it) and lets its slots be evicted again.
int cache_release(moe_expert_cache* c, int layer, cudaStream_t compute);

// ---- copy kernels and the device-side LRU (cache_dev.cu)
// Builds d_src, the device table of the host bundles' device-visible addresses.
int cache_src_init(moe_expert_cache* c);
// Enqueues on the copy stream one kernel that copies bundle keys[j] (layer * E + expert) from
// the host store into slot slots[j], j < n <= kMaxExperts (needs d_src).
int cache_fill_slots(moe_expert_cache* c, int n, const int32_t* keys, const int32_t* slots);
enum DevCtl { kClock = 0, kReq, kTraceN, kOverflow, kHits, kMisses, kEvictions, kBytes, kDevCtl = 16 };
// Allocates and initialises the device state (empty cache).
int cache_dev_init(moe_expert_cache* c);
void cache_dev_free(moe_expert_cache* c);
// Enqueues, for `layer`, the LRU request over the experts with counts[e] > 0 (device [E]) on
// stream `s0`, and the copies of its misses on the cache's copy stream (joined back later by
// cache_dev_wait_copies).  Fills d_ptrs and the hit / miss lists.  A request that needs more
// distinct bundles than slots records MOE_ERR_CAPACITY in *err and leaves the state alone.
int cache_dev_request(moe_expert_cache* c, int layer, const int32_t* counts, cudaStream_t s0,
                      int32_t* err);
int cache_dev_wait_copies(moe_expert_cache* c, cudaStream_t s0);
// Device lists of the latest request.
inline const int32_t* dev_hit_list(const moe_expert_cache* c) { return c->d_lists; }
inline const int32_t* dev_n_hit(const moe_expert_cache* c) { return c->d_lists + c->E; }
inline const int32_t* dev_miss_list(const moe_expert_cache* c) { return c->d_lists + c->E + 1; }
inline const int32_t* dev_n_miss(const moe_expert_cache* c) { return c->d_lists + 3 * c->E + 1; }
}  // namespace moe

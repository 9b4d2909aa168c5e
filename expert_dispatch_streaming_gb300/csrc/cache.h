// Expert-slot cache internals shared by cache.cpp and the layer forward (internal).
#pragma once
#include <cuda_runtime.h>

#include <list>
#include <set>
#include <unordered_map>
#include <vector>

#include "../../include/moe.h"

struct moe_expert_cache {
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
  std::vector<char> slot_pending;        // filled, and no compute has waited for it yet
  std::vector<char> slot_prefetched;     // filled by a prefetch, not yet used by a request
  int prefetch_next = 0;
  std::vector<moe_cache_event> trace;
  moe_cache_stats st{};
  long long req = 0;
  // copy timing (time_copies): event pairs of copies not yet collected, and a free pool
  int time_copies = 0;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> timed, pool;
};

namespace moe {
int cache_wait_event(moe_expert_cache* c, cudaEvent_t ev);
// Request with the hit/miss split reported (used by the layer forward).  wait_slots (nullable)
// receives the slots of hits whose copy (a prefetch) no compute has waited for yet; the caller
// makes its compute stream wait on their ready events before using them.
int cache_request_split(moe_expert_cache* c, int layer, const uint8_t* used, cudaStream_t compute,
                        const void** slot_ptrs, std::vector<int>* hits, std::vector<int>* misses,
                        std::vector<int>* wait_slots = nullptr);
// Prefetch request (see moe_expert_cache_prefetch); mask NULL = the layer's last expert set.
int cache_prefetch(moe_expert_cache* c, int layer, const uint8_t* mask, int32_t* n_filled);
}  // namespace moe

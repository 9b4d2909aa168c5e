// moe_route_topk_static: the routing call for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or pass a workspace: a plug-in running inside a host
// framework that owns all device memory and forbids allocations of its own, or code on a
// latency-critical path where an allocation (and the device-wide synchronisation cudaFree can
// cause) is not acceptable.  This entry point routes exactly like moe_route_topk, but its
// scratch lives in a fixed array in the library's own device memory instead of a caller
// workspace.
//
// The array is a file-scope __device__ variable, so every GPU that loads the library holds it
// until the process exits.  In host code its name is only a host-side stand-in for the device
// variable, not a device address: the first call on each device, with that device current,
// looks the real address up with cudaGetSymbolAddress and keeps it for later calls.  The kept
// address belongs to the device's primary context: after cudaDeviceReset (or anything else that
// destroys and recreates that context) it is stale, so these entry points must not be used
// across a device reset.
#include <mutex>

#include "common.cuh"
#include "route.cuh"

namespace moe {
namespace {

// Largest routing scratch this entry point serves (8 MiB, per device).
constexpr size_t kStaticRouteScratchBytes = size_t(8) << 20;

static __device__ __align__(256) unsigned char g_route_scratch[kStaticRouteScratchBytes];

constexpr int kMaxDevices = 128;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once per device).
int static_scratch(void** out) {
  int dev = -1;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t r = cudaGetSymbolAddress(&p, g_route_scratch);
    if (r != cudaSuccess || !p) return fail_cuda(r != cudaSuccess ? r : cudaErrorInvalidSymbol);
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_route_topk_static(const uint16_t* x, const float* w_r, const float* logit_bias,
                                     const float* sel_bias, const uint16_t* w_gate,
                                     const int32_t* forced_ids, int T, int H, int E, int k,
                                     int gating, float scale, int32_t* ids, float* w,
                                     int32_t* counts, int32_t* offsets, int32_t* pos,
                                     int32_t* src, float* logits, float* shared_gate,
                                     int32_t* tie_flags, void* stream) {
  const size_t need = moe_route_workspace_size(T, H, E, k);
  if (need == 0) return MOE_ERR_INVALID_ARG;
  if (need > moe::kStaticRouteScratchBytes) return MOE_ERR_CAPACITY;
  void* scratch = nullptr;
  const int r = moe::static_scratch(&scratch);
  if (r != MOE_OK) return r;
  // Every byte of routing scratch that must start at zero (the per-tile histogram) is cleared
  // by the routing kernels themselves at the start of each call.
  return moe_route_topk(x, w_r, logit_bias, sel_bias, w_gate, forced_ids, T, H, E, k, gating,
                        scale, ids, w, counts, offsets, pos, src, logits, shared_gate,
                        tie_flags, scratch, moe::kStaticRouteScratchBytes, stream);
}

extern "C" int moe_route_static_error(int32_t* code, void* stream) {
  if (!code) return MOE_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const int r = moe::static_scratch(&scratch);
  if (r != MOE_OK) return r;
  // moe_route_topk keeps its error word in the first 4 bytes of its scratch
  return moe_workspace_error(scratch, code, stream);
}

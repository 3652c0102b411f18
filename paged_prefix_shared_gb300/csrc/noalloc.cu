// pps_attn_run_noalloc: the mixed-batch attention for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at all: a plugin loaded into an engine
// that owns every byte of device memory and hands plugins no workspace, or a
// latency-critical loop that must never reach cudaMalloc / cudaFree (both can
// synchronize the whole device).  pps_attn_run needs a caller-supplied
// workspace for the task table and the fp32 partials; this entry point uses a
// fixed-size array that the library itself places in device memory instead.
//
// The array lives at file scope below.  Every GPU that loads this library
// holds it (PPS_NOALLOC_SCRATCH_BYTES) until the process exits.  Host code
// cannot use the array's name as a device address (on the host it is only a
// stand-in symbol), so the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current and caches it.
#include <cuda_runtime.h>

#include <mutex>

#include "pps_internal.h"

namespace {

static __device__ __align__(256) uint8_t g_pps_noalloc_scratch[PPS_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device; looked up once
// per device (this is the set-up the first call on a device performs).
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pps_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" pps_status pps_attn_run_noalloc(const pps_plan* plan, const void* q,
                                           const pps_pool* pool, void* out, void* stream) {
  if (!plan) return PPS_ERR_INVALID_ARGUMENT;
  if (plan->workspace_bytes > (size_t)PPS_NOALLOC_SCRATCH_BYTES) return PPS_ERR_SCRATCH_LIMIT;
  void* ws = scratch_address();
  if (!ws) return PPS_ERR_CUDA;
  // Same work as pps_attn_run, with the library's own array as the workspace.
  // Nothing in it has to start at zero: each call uploads its task table first
  // and every partial a kernel reads was written earlier in the same call.
  return pps_attn_run(plan, q, pool, out, ws, (size_t)PPS_NOALLOC_SCRATCH_BYTES, stream);
}

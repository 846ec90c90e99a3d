// tt_forward_noalloc: the forward of one TT layer for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain device scratch: a plain-C host or
// plugin that owns no CUDA allocator of its own, or a process whose policy
// forbids cudaMalloc once it is running (allocation can stall, fragment the
// heap or fail at a bad moment in a long-running or latency-bound service).
// For them the scratch that tt_forward normally takes from the caller lives
// in a fixed, file-scope device array of this library instead.
//
// Costs and rules:
//  - every GPU that loads this library holds kNoAllocScratchBytes (32 MiB)
//    of device memory for the array until the process exits;
//  - the first call on a device looks the array's device address up
//    (cudaGetSymbolAddress, once per device, with that device current), so
//    make that first call before any stream capture;
//  - all calls share the one array and it keeps the last call's contents:
//    calls whose work overlaps on the GPU (different streams, or a second
//    call before the first finished on another stream) race on it;
//  - nothing in the array has to start at zero: the forward writes every
//    scratch byte before it reads it.
#include <cuda_runtime.h>

#include <mutex>

#include "ttc.h"
#include "ttc_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

extern "C" tt_status tt_forward_noalloc(const tt_plan_t* plan, int64_t T, const void* x,
                                        const float* params, void* y, void* stream) {
  if (!plan || plan->kind != 0 || T < 0) return TT_ERR_INVALID_ARG;
  size_t need = 0;
  tt_status s = tt_workspace_size(plan, T, &need);
  if (s != TT_OK) return s;
  if (need > kNoAllocScratchBytes) return TT_ERR_WORKSPACE;
  if (T == 0) return TT_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TT_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TT_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return TT_ERR_CUDA;
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  return tt_forward(plan, T, x, params, y, scratch, kNoAllocScratchBytes, stream);
}

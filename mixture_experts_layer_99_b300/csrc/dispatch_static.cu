// Dispatch for callers that cannot provide a workspace.
//
// moe_dispatch needs scratch memory for its per-block expert histograms and
// their scanned bases, and takes it from a caller-allocated workspace. Some
// callers cannot allocate one: a plugin or custom-op interface that hands the
// op only its own input and output tensors, or a runtime that fixes its
// device memory map at start-up and forbids cudaMalloc afterwards. This entry
// point takes its scratch from a fixed array in the library's own device
// memory instead, and allocates nothing.
#include "moe_internal.h"

#include <mutex>

namespace moe {
namespace {

// Entries per scratch array (histograms, then bases): blocks * E must fit.
constexpr int64_t kStaticScratchEntries = 65536;
constexpr int kMaxDevices = 64;

// 2 x 65536 int32 = 512 KiB, loaded with the library on every device that
// uses it and held until the process exits.
__device__ __align__(256) int32_t g_dispatch_scratch[2 * kStaticScratchEntries];

// The array's device address on each device, once a lookup has succeeded
// (a failed lookup is not kept: the next call tries again).
struct DeviceScratch {
  std::mutex mu;
  int32_t* ptr = nullptr;
};
DeviceScratch g_scratch[kMaxDevices];

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_dispatch_static_scratch(const moe_config_t* cfg,
                                                    const int32_t* topk_idx, const void* x,
                                                    int32_t* expert_count,
                                                    int32_t* expert_offset, int32_t* slot_of,
                                                    int32_t* token_of_row, void* xd,
                                                    moe_stream_t stream) {
  using namespace moe;
  size_t unused = 0;
  const moe_status_t st = moe_workspace_size(cfg, &unused);  // validates cfg
  if (st != MOE_OK) return st;
  if (!topk_idx || !x || !expert_count || !expert_offset || !slot_of || !token_of_row || !xd)
    return MOE_ERR_INVALID_ARG;
  const int64_t nblk = disp_blocks(*cfg);
  if (nblk * cfg->E > kStaticScratchEntries) return MOE_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  DeviceScratch& ds = g_scratch[dev];
  // First call on this device (with it current): host code cannot use the
  // array's name as a device address, so look the address up; it is kept
  // only once a lookup has succeeded.
  int32_t* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(ds.mu);
    if (ds.ptr == nullptr) {
      int32_t* p = nullptr;
      if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_dispatch_scratch) == cudaSuccess)
        ds.ptr = p;
      else
        (void)cudaGetLastError();  // do not leave the failure for a later launch check
    }
    scratch = ds.ptr;
  }
  if (scratch == nullptr) return MOE_ERR_CUDA;
  // Both arrays are fully rewritten by every call (histograms by the count
  // kernel, bases by the scan kernel), so nothing needs clearing first.
  const cudaError_t e = launch_dispatch(*cfg, topk_idx, x, expert_count, expert_offset, slot_of,
                                        token_of_row, xd, scratch, scratch + kStaticScratchEntries,
                                        (int64_t)cfg->T * cfg->k, (cudaStream_t)stream);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

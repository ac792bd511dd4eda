// ep_get_layout_noalloc: the layout for callers that cannot allocate device
// memory.  The layout kernels need scratch memory for their per-tile
// histograms (the `workspace` of ep_get_layout).  Some callers have no way
// to provide it: code running inside a host framework that owns every byte
// of device memory and hands out no extra buffers, a serving loop that must
// not allocate once it has warmed up (cudaMalloc can synchronise the device
// and fragment a carefully sized pool), or a plugin whose interface only
// passes the tensors it computes on.  For them the scratch lives in this
// library's own device memory: a fixed-size array defined below, which every
// GPU that loads the library holds until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/ep.h"
#include "ep_internal.h"

namespace ep {

// Largest scratch the allocation-free entry point can offer.
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB

// The scratch itself.  In host code this name is only a stand-in for the
// device array; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_layout_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxScratchDevices = 64;

struct ScratchSlot {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t status = cudaSuccess;
};

ScratchSlot g_slots[kMaxScratchDevices];

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
int32_t scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices)
    return EP_ERR_CUDA;
  ScratchSlot& slot = g_slots[dev];
  std::call_once(slot.once, [&slot] {
    void* p = nullptr;
    slot.status = cudaGetSymbolAddress(&p, g_layout_scratch);
    slot.ptr = slot.status == cudaSuccess ? p : nullptr;
  });
  if (slot.status != cudaSuccess || slot.ptr == nullptr) return EP_ERR_CUDA;
  *out = slot.ptr;
  return EP_OK;
}

}  // namespace
}  // namespace ep

extern "C" int32_t ep_get_layout_noalloc(const ep_config* cfg, int32_t num_tokens,
                                         const int64_t* d_topk_idx,
                                         ep_layout* layout,
                                         int32_t* h_expert_count, void* stream) {
  if (cfg == nullptr || layout == nullptr) return EP_ERR_INVALID_ARG;
  const int64_t need = ep_layout_workspace_bytes(cfg);
  if (need < 0) return EP_ERR_INVALID_ARG;
  // only the two-launch layout uses the scratch
  if (need > static_cast<int64_t>(ep::kNoAllocScratchBytes) &&
      !ep::layout_is_small(num_tokens, cfg->num_topk, cfg->num_experts))
    return EP_ERR_CAPACITY;
  void* scratch = nullptr;
  const int32_t st = ep::scratch_address(&scratch);
  if (st != EP_OK) return st;
  // Same launches as ep_get_layout, with the workspace taken from the
  // library's array instead of from the caller.
  ep_layout with_scratch = *layout;
  with_scratch.workspace = scratch;
  const int32_t rc = ep_get_layout(cfg, num_tokens, d_topk_idx, &with_scratch,
                                   h_expert_count, stream);
  layout->num_tokens = with_scratch.num_tokens;
  return rc;
}

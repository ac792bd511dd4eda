// extern "C" entry points of libep_gb300.so (declared in include/ep.h):
// host-side validation, sizing, and launches on the caller's stream.  The
// library holds no state besides a per-device property cache and, once the
// host-buffer entry points have copied in chunks on a device, that device's
// two copy streams (one a direction) and their events.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/ep.h"
#include "ep_device.cuh"
#include "ep_internal.h"

namespace ep {

constexpr int kMaxDevices = 64;

const DeviceInfo& device_info() {
  static DeviceInfo infos[kMaxDevices];
  static std::once_flag once[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
  std::call_once(once[dev], [dev] {
    DeviceInfo& d = infos[dev];
    d.sm_count = 1;
    d.max_smem_optin = 48 * 1024;
    d.smem_per_sm = 48 * 1024;
    cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  });
  return infos[dev];
}

static thread_local cudaError_t g_last_cuda_error = cudaSuccess;

cudaError_t note_cuda(cudaError_t e) {
  if (e != cudaSuccess) g_last_cuda_error = e;
  return e;
}

// One-time per-device kernel set-up (shared-memory limits).
static cudaError_t ensure_prepared() {
  static std::once_flag once[kMaxDevices];
  static cudaError_t result[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
  std::call_once(once[dev], [dev] {
    (void)device_info();
    cudaError_t e = prepare_layout_kernels();
    if (e == cudaSuccess) e = prepare_dispatch_kernels();
    result[dev] = e;
  });
  return note_cuda(result[dev]);
}

static bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

static bool config_ok(const ep_config* c) {
  if (c == nullptr) return false;
  if (c->max_tokens < 0 || c->hidden < 8 || c->hidden % 8 != 0) return false;
  if (c->hidden > (1 << 20)) return false;
  if (c->num_topk < 1 || c->num_topk > 32) return false;
  if (c->num_experts < 1 || c->num_experts > 2048) return false;
  if (c->num_topk > c->num_experts) return false;
  if (c->num_ranks < 1 || c->num_ranks > c->num_experts) return false;
  if (c->num_experts % c->num_ranks != 0) return false;
  if (c->expert_alignment < 1 || c->expert_alignment > 1024) return false;
  if (c->use_fp8_dispatch != 0 && c->use_fp8_dispatch != 1) return false;
  if (c->zero_padding != 0 && c->zero_padding != 1) return false;
  if (c->use_fp8_dispatch && c->hidden % 128 != 0) return false;
  // bf16 rows: up to the widest row the GPU parity cases cover
  // all row indices fit in int32
  const int64_t cap = int64_t(c->max_tokens) * c->num_topk +
                      int64_t(c->num_experts) * (c->expert_alignment - 1);
  if (cap >= (int64_t(1) << 31)) return false;
  return true;
}

static int64_t capacity(const ep_config* c) {
  return int64_t(c->max_tokens) * c->num_topk +
         int64_t(c->num_experts) * (c->expert_alignment - 1);
}

static int32_t cuda_status(cudaError_t e) {
  return note_cuda(e) == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

static int32_t status_from_bits(int32_t bits) {
  if (bits & ERRBIT_EXPERT_RANGE) return EP_ERR_EXPERT_RANGE;
  if (bits & ERRBIT_DUP_EXPERT) return EP_ERR_DUP_EXPERT;
  if (bits & ERRBIT_TIMEOUT_PENDING) return EP_ERR_TIMEOUT_PENDING;
  if (bits & ERRBIT_TIMEOUT) return EP_ERR_TIMEOUT;
  return EP_OK;
}

static bool layout_ptrs_ok(const ep_layout* L) {
  if (L == nullptr) return false;
  const void* ps[] = {L->expert_count, L->expert_start, L->expert_end,
                      L->rank_start, L->tokens_per_rank, L->is_token_in_rank,
                      L->slot_of, L->src_info, L->err, L->workspace};
  for (const void* p : ps)
    if (p == nullptr || !aligned16(p)) return false;
  // optional rank rows: all three or none
  const void* rs[] = {L->rank_row_start, L->rank_slot_of, L->rank_src};
  const int set = (rs[0] != nullptr) + (rs[1] != nullptr) + (rs[2] != nullptr);
  if (set != 0 && set != 3) return false;
  for (const void* p : rs)
    if (p != nullptr && !aligned16(p)) return false;
  return true;
}

static bool has_rank_rows(const ep_layout* L) { return L->rank_slot_of != nullptr; }

static int64_t rank_rows_capacity(const ep_config* c) {
  const int per = c->num_topk < c->num_ranks ? c->num_topk : c->num_ranks;
  return int64_t(c->max_tokens) * per;
}

}  // namespace ep

using namespace ep;

extern "C" {

int64_t ep_recv_capacity(const ep_config* cfg) {
  return config_ok(cfg) ? capacity(cfg) : -1;
}

int64_t ep_layout_workspace_bytes(const ep_config* cfg) {
  if (!config_ok(cfg)) return -1;
  return layout_workspace_bytes(cfg->num_experts, cfg->num_ranks);
}

// Checks the arguments of a layout call and fills its launch arguments.
static int32_t layout_args(const ep_config* cfg, int32_t num_tokens,
                           const int64_t* d_topk_idx, const ep_layout* layout, LayoutArgs* a) {
  if (!config_ok(cfg) || !layout_ptrs_ok(layout)) return EP_ERR_INVALID_ARG;
  if (num_tokens < 0 || num_tokens > cfg->max_tokens) return EP_ERR_INVALID_ARG;
  if (num_tokens > 0 && (d_topk_idx == nullptr || !aligned16(d_topk_idx)))
    return EP_ERR_INVALID_ARG;
  const int K = cfg->num_topk, E = cfg->num_experts, R = cfg->num_ranks;
  a->topk_idx = d_topk_idx;
  a->T = num_tokens;
  a->K = K;
  a->E = E;
  a->R = R;
  a->A = cfg->expert_alignment;
  a->geom = layout_tiles(num_tokens > 0 ? num_tokens : 1, K);
  if (a->geom.num_tiles > kLayoutMaxTiles) return EP_ERR_INVALID_ARG;
  a->ws = carve_layout_workspace(layout->workspace, E, R);
  a->expert_count = layout->expert_count;
  a->expert_start = layout->expert_start;
  a->expert_end = layout->expert_end;
  a->rank_start = layout->rank_start;
  a->tokens_per_rank = layout->tokens_per_rank;
  a->slot_of = layout->slot_of;
  a->src_info = layout->src_info;
  a->err = layout->err;
  a->is_token_in_rank = layout->is_token_in_rank;
  a->rank_row_start = layout->rank_row_start;
  a->rank_slot_of = layout->rank_slot_of;
  a->rank_src = layout->rank_src;
  return EP_OK;
}

int32_t ep_get_layout(const ep_config* cfg, int32_t num_tokens,
                      const int64_t* d_topk_idx, ep_layout* layout,
                      int32_t* h_expert_count, void* stream) {
  LayoutArgs a;
  const int32_t v = layout_args(cfg, num_tokens, d_topk_idx, layout, &a);
  if (v != EP_OK) return v;
  if (ensure_prepared() != cudaSuccess) return EP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = note_cuda(launch_layout(a, s));
  if (e != cudaSuccess) return EP_ERR_CUDA;
  layout->num_tokens = num_tokens;
  if (h_expert_count != nullptr) {
    int32_t bits = 0;
    e = cudaMemcpyAsync(h_expert_count, layout->expert_count, sizeof(int32_t) * a.E,
                        cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(&bits, layout->err, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (note_cuda(e) != cudaSuccess) return EP_ERR_CUDA;
    return status_from_bits(bits);
  }
  return EP_OK;
}

// Checks the arguments of a dispatch of T tokens and fills its launch
// arguments.
static int32_t dispatch_args(const ep_config* cfg, const ep_layout* layout, int T,
                             const void* d_x, const float* d_topk_weights, void* d_recv_x,
                             float* d_recv_scale, float* d_recv_w, DispatchArgs* a) {
  if (!config_ok(cfg) || !layout_ptrs_ok(layout)) return EP_ERR_INVALID_ARG;
  if (T < 0 || T > cfg->max_tokens) return EP_ERR_INVALID_ARG;
  if (d_recv_x == nullptr || !aligned16(d_recv_x)) return EP_ERR_INVALID_ARG;
  if (T > 0 && (d_x == nullptr || !aligned16(d_x))) return EP_ERR_INVALID_ARG;
  if (d_topk_weights != nullptr && !aligned16(d_topk_weights)) return EP_ERR_INVALID_ARG;
  if (d_recv_w != nullptr && !aligned16(d_recv_w)) return EP_ERR_INVALID_ARG;
  if (d_recv_w != nullptr && d_topk_weights == nullptr) return EP_ERR_INVALID_ARG;
  if (cfg->use_fp8_dispatch && (d_recv_scale == nullptr || !aligned16(d_recv_scale)))
    return EP_ERR_INVALID_ARG;
  a->x = d_x;
  a->topk_weights = d_topk_weights;
  a->slot_of = layout->slot_of;
  a->expert_start = layout->expert_start;
  a->expert_end = layout->expert_end;
  a->T = T;
  a->H = cfg->hidden;
  a->K = cfg->num_topk;
  a->E = cfg->num_experts;
  a->fp8 = cfg->use_fp8_dispatch != 0;
  a->zero_padding = cfg->zero_padding != 0;
  a->recv_x = d_recv_x;
  a->recv_scale = d_recv_scale;
  a->recv_w = d_recv_w;
  a->err = layout->err;
  return EP_OK;
}

int32_t ep_dispatch(const ep_config* cfg, const ep_layout* layout,
                    const void* d_x, const float* d_topk_weights,
                    void* d_recv_x, float* d_recv_scale, float* d_recv_w,
                    void* stream) {
  if (layout == nullptr) return EP_ERR_INVALID_ARG;
  DispatchArgs a;
  const int32_t v = dispatch_args(cfg, layout, layout->num_tokens, d_x, d_topk_weights,
                                  d_recv_x, d_recv_scale, d_recv_w, &a);
  if (v != EP_OK) return v;
  if (ensure_prepared() != cudaSuccess) return EP_ERR_CUDA;
  return cuda_status(launch_dispatch(a, static_cast<cudaStream_t>(stream)));
}

int32_t ep_layout_and_dispatch(const ep_config* cfg, int32_t num_tokens,
                               const int64_t* d_topk_idx, ep_layout* layout,
                               const void* d_x, const float* d_topk_weights,
                               void* d_recv_x, float* d_recv_scale, float* d_recv_w,
                               void* stream) {
  LayoutArgs la;
  int32_t v = layout_args(cfg, num_tokens, d_topk_idx, layout, &la);
  if (v != EP_OK) return v;
  DispatchArgs da;
  v = dispatch_args(cfg, layout, num_tokens, d_x, d_topk_weights, d_recv_x, d_recv_scale,
                    d_recv_w, &da);
  if (v != EP_OK) return v;
  if (ensure_prepared() != cudaSuccess) return EP_ERR_CUDA;
  const cudaError_t e = note_cuda(launch_layout_dispatch(la, da, static_cast<cudaStream_t>(stream)));
  if (e != cudaSuccess) return EP_ERR_CUDA;
  layout->num_tokens = num_tokens;
  return EP_OK;
}

int32_t ep_combine(const ep_config* cfg, const ep_layout* layout,
                   const void* d_expert_out, const float* d_topk_weights,
                   void* d_y, void* stream) {
  if (!config_ok(cfg) || !layout_ptrs_ok(layout)) return EP_ERR_INVALID_ARG;
  const int T = layout->num_tokens;
  if (T < 0 || T > cfg->max_tokens) return EP_ERR_INVALID_ARG;
  if (T > 0) {
    if (d_expert_out == nullptr || !aligned16(d_expert_out)) return EP_ERR_INVALID_ARG;
    if (d_y == nullptr || !aligned16(d_y)) return EP_ERR_INVALID_ARG;
  }
  if (d_topk_weights != nullptr && !aligned16(d_topk_weights)) return EP_ERR_INVALID_ARG;
  if (ensure_prepared() != cudaSuccess) return EP_ERR_CUDA;
  CombineArgs a;
  a.expert_out = d_expert_out;
  a.topk_weights = d_topk_weights;
  a.slot_of = layout->slot_of;
  a.T = T;
  a.H = cfg->hidden;
  a.K = cfg->num_topk;
  a.y = d_y;
  return cuda_status(launch_combine(a, static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------------------
// host buffers: copies in token chunks overlapped with the row kernels
// ---------------------------------------------------------------------------
constexpr int kMaxHostChunks = 64;

// Per device and per copy direction (host to device for
// ep_dispatch_from_host, device to host for ep_combine_to_host): one copy
// stream and kMaxHostChunks + 1 events, created by the first host-buffer
// call on the device and kept until exit.  With a stream per direction, a
// combine's rows going out and the next batch's rows coming in (two calls on
// two streams) run on the two copy engines at once.
struct HostIoLane {
  cudaStream_t copy = nullptr;
  cudaEvent_t ev[kMaxHostChunks + 1] = {};
};
struct HostIo {
  HostIoLane h2d, d2h;
};

static cudaError_t host_io(HostIo** out) {
  static HostIo io[kMaxDevices];
  static std::once_flag once[kMaxDevices];
  static cudaError_t result[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
  std::call_once(once[dev], [dev] {
    cudaError_t e = cudaSuccess;
    for (HostIoLane* lane : {&io[dev].h2d, &io[dev].d2h}) {
      if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&lane->copy, cudaStreamNonBlocking);
      for (int i = 0; e == cudaSuccess && i <= kMaxHostChunks; ++i)
        e = cudaEventCreateWithFlags(&lane->ev[i], cudaEventDisableTiming);
    }
    result[dev] = e;
  });
  *out = &io[dev];
  return note_cuda(result[dev]);
}

// Rows a chunk carries at least: each chunk costs a few µs of copy start-up
// and cross-stream signalling, which pays off only on copies of several MB.
constexpr int64_t kMinChunkBytes = int64_t(4) << 20;

// Tokens per chunk: T split into at most `chunks` chunks of at least
// kMinChunkBytes each, ceil(T / n) tokens a chunk, the last ragged.
static int chunk_tokens(int T, int chunks, int64_t row_bytes) {
  int64_t n = int64_t(T) * row_bytes / kMinChunkBytes;
  if (n > chunks) n = chunks;
  if (n < 1) n = 1;
  return int((T + n - 1) / n);
}

// The device address of page-locked host memory (cudaHostAlloc, or
// cudaHostRegister with mapping), 16-byte aligned; nullptr for anything else.
static void* mapped_host(const void* h) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, h) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) return nullptr;
  return aligned16(attr.devicePointer) ? attr.devicePointer : nullptr;
}

int32_t ep_dispatch_from_host(const ep_config* cfg, const ep_layout* layout,
                              const void* h_x, void* d_x, const float* d_topk_weights,
                              void* d_recv_x, float* d_recv_scale, float* d_recv_w,
                              int32_t num_chunks, void* stream) {
  if (!config_ok(cfg) || !layout_ptrs_ok(layout)) return EP_ERR_INVALID_ARG;
  const int T = layout->num_tokens;
  if (T < 0 || T > cfg->max_tokens) return EP_ERR_INVALID_ARG;
  if (num_chunks < 0 || num_chunks > kMaxHostChunks) return EP_ERR_INVALID_ARG;
  if (d_recv_x == nullptr || !aligned16(d_recv_x)) return EP_ERR_INVALID_ARG;
  const bool direct = num_chunks == 0;
  if (T > 0 && (h_x == nullptr || (!direct && (d_x == nullptr || !aligned16(d_x)))))
    return EP_ERR_INVALID_ARG;
  const void* x_mapped = direct && T > 0 ? mapped_host(h_x) : nullptr;
  if (direct && T > 0 && x_mapped == nullptr) return EP_ERR_INVALID_ARG;
  if (d_topk_weights != nullptr && !aligned16(d_topk_weights)) return EP_ERR_INVALID_ARG;
  if (d_recv_w != nullptr && !aligned16(d_recv_w)) return EP_ERR_INVALID_ARG;
  if (d_recv_w != nullptr && d_topk_weights == nullptr) return EP_ERR_INVALID_ARG;
  if (cfg->use_fp8_dispatch && (d_recv_scale == nullptr || !aligned16(d_recv_scale)))
    return EP_ERR_INVALID_ARG;
  if (ensure_prepared() != cudaSuccess) return EP_ERR_CUDA;
  HostIo* io = nullptr;
  if (!direct && host_io(&io) != cudaSuccess) return EP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int K = cfg->num_topk;
  const int64_t row_bytes = int64_t(cfg->hidden) * 2;
  DispatchArgs base;
  base.topk_weights = d_topk_weights;
  base.slot_of = layout->slot_of;
  base.expert_start = layout->expert_start;
  base.expert_end = layout->expert_end;
  base.H = cfg->hidden;
  base.K = K;
  base.E = cfg->num_experts;
  base.fp8 = cfg->use_fp8_dispatch != 0;
  base.zero_padding = false;
  base.recv_x = d_recv_x;
  base.recv_scale = d_recv_scale;
  base.recv_w = d_recv_w;
  base.err = layout->err;
  base.pdl = false;
  cudaError_t e = cudaSuccess;
  const int tc = T > 0 && !direct ? chunk_tokens(T, num_chunks, row_bytes) : 0;
  if (direct && T > 0) {
    // the kernel reads the rows where they are, once, over the host link
    DispatchArgs a = base;
    a.x = x_mapped;
    a.T = T;
    a.pdl = true;
    e = launch_dispatch(a, s);
  } else if (T > 0 && tc >= T) {
    // one chunk: the copy and the kernel in order on the caller's stream
    e = cudaMemcpyAsync(d_x, h_x, T * row_bytes, cudaMemcpyHostToDevice, s);
    DispatchArgs a = base;
    a.x = d_x;
    a.T = T;
    if (e == cudaSuccess) e = launch_dispatch(a, s);
  } else if (T > 0) {
    const int n_chunks = (T + tc - 1) / tc;
    // the staging rows are free once the stream's earlier work is done
    HostIoLane* io_in = &io->h2d;
    e = cudaEventRecord(io_in->ev[kMaxHostChunks], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(io_in->copy, io_in->ev[kMaxHostChunks], 0);
    for (int c = 0; e == cudaSuccess && c < n_chunks; ++c) {
      const int t0 = c * tc, n = T - t0 < tc ? T - t0 : tc;
      e = cudaMemcpyAsync(static_cast<char*>(d_x) + t0 * row_bytes,
                          static_cast<const char*>(h_x) + t0 * row_bytes, n * row_bytes,
                          cudaMemcpyHostToDevice, io_in->copy);
      if (e == cudaSuccess) e = cudaEventRecord(io_in->ev[c], io_in->copy);
    }
    for (int c = 0; e == cudaSuccess && c < n_chunks; ++c) {
      const int t0 = c * tc, n = T - t0 < tc ? T - t0 : tc;
      e = cudaStreamWaitEvent(s, io_in->ev[c], 0);
      if (e != cudaSuccess) break;
      DispatchArgs a = base;
      a.x = static_cast<const char*>(d_x) + t0 * row_bytes;
      a.topk_weights = d_topk_weights != nullptr ? d_topk_weights + int64_t(t0) * K : nullptr;
      a.slot_of = layout->slot_of + int64_t(t0) * K;
      a.T = n;
      e = launch_dispatch(a, s);
    }
  }
  if (e == cudaSuccess && cfg->zero_padding) {
    DispatchArgs z = base;
    z.T = 0;
    z.zero_padding = true;
    e = launch_dispatch(z, s);
  }
  return cuda_status(e);
}

int32_t ep_combine_to_host(const ep_config* cfg, const ep_layout* layout,
                           const void* d_expert_out, const float* d_topk_weights,
                           void* d_y, void* h_y, int32_t num_chunks, void* stream) {
  if (!config_ok(cfg) || !layout_ptrs_ok(layout)) return EP_ERR_INVALID_ARG;
  const int T = layout->num_tokens;
  if (T < 0 || T > cfg->max_tokens) return EP_ERR_INVALID_ARG;
  if (num_chunks < 0 || num_chunks > kMaxHostChunks) return EP_ERR_INVALID_ARG;
  const bool direct = num_chunks == 0;
  if (T > 0) {
    if (d_expert_out == nullptr || !aligned16(d_expert_out)) return EP_ERR_INVALID_ARG;
    if (h_y == nullptr || (!direct && (d_y == nullptr || !aligned16(d_y))))
      return EP_ERR_INVALID_ARG;
  }
  if (d_topk_weights != nullptr && !aligned16(d_topk_weights)) return EP_ERR_INVALID_ARG;
  if (T == 0) return EP_OK;
  void* y_mapped = direct ? mapped_host(h_y) : nullptr;
  if (direct && y_mapped == nullptr) return EP_ERR_INVALID_ARG;
  if (ensure_prepared() != cudaSuccess) return EP_ERR_CUDA;
  if (direct) {
    // the kernel writes the rows where they belong, once, over the host link
    CombineArgs a;
    a.expert_out = d_expert_out;
    a.topk_weights = d_topk_weights;
    a.slot_of = layout->slot_of;
    a.T = T;
    a.H = cfg->hidden;
    a.K = cfg->num_topk;
    a.y = y_mapped;
    return cuda_status(launch_combine(a, static_cast<cudaStream_t>(stream)));
  }
  HostIo* io = nullptr;
  if (host_io(&io) != cudaSuccess) return EP_ERR_CUDA;
  HostIoLane* io_out = &io->d2h;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int K = cfg->num_topk;
  const int64_t row_bytes = int64_t(cfg->hidden) * 2;
  const int tc = chunk_tokens(T, num_chunks, row_bytes);
  const int n_chunks = (T + tc - 1) / tc;
  cudaError_t e = cudaSuccess;
  if (n_chunks == 1) {
    // one chunk: the kernel and the copy in order on the caller's stream
    CombineArgs a;
    a.expert_out = d_expert_out;
    a.topk_weights = d_topk_weights;
    a.slot_of = layout->slot_of;
    a.T = T;
    a.H = cfg->hidden;
    a.K = K;
    a.y = d_y;
    e = launch_combine(a, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h_y, d_y, T * row_bytes, cudaMemcpyDeviceToHost, s);
    return cuda_status(e);
  }
  for (int c = 0; e == cudaSuccess && c < n_chunks; ++c) {
    const int t0 = c * tc, n = T - t0 < tc ? T - t0 : tc;
    CombineArgs a;
    a.expert_out = d_expert_out;
    a.topk_weights = d_topk_weights != nullptr ? d_topk_weights + int64_t(t0) * K : nullptr;
    a.slot_of = layout->slot_of + int64_t(t0) * K;
    a.T = n;
    a.H = cfg->hidden;
    a.K = K;
    a.y = static_cast<char*>(d_y) + t0 * row_bytes;
    a.pdl = false;
    e = launch_combine(a, s);
    if (e == cudaSuccess) e = cudaEventRecord(io_out->ev[c], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(io_out->copy, io_out->ev[c], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<char*>(h_y) + t0 * row_bytes,
                          static_cast<const char*>(d_y) + t0 * row_bytes, n * row_bytes,
                          cudaMemcpyDeviceToHost, io_out->copy);
  }
  // the caller's stream completes only after the last rows reached the host
  if (e == cudaSuccess) e = cudaEventRecord(io_out->ev[kMaxHostChunks], io_out->copy);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, io_out->ev[kMaxHostChunks], 0);
  return cuda_status(e);
}

int64_t ep_scale_ld(const ep_config* cfg) {
  if (!config_ok(cfg)) return -1;
  return (capacity(cfg) + 3) / 4 * 4;
}

int32_t ep_dispatch_fp8(const ep_config* cfg, const ep_layout* layout,
                        const void* d_x, const uint8_t* d_x_q,
                        const float* d_x_scale, const float* d_topk_weights,
                        uint8_t* d_recv_q, float* d_recv_scale,
                        int32_t scale_col_major, float* d_recv_w, void* stream) {
  if (!config_ok(cfg) || !layout_ptrs_ok(layout)) return EP_ERR_INVALID_ARG;
  if (cfg->hidden % 128 != 0) return EP_ERR_INVALID_ARG;
  if (scale_col_major != 0 && scale_col_major != 1) return EP_ERR_INVALID_ARG;
  const int T = layout->num_tokens;
  if (T < 0 || T > cfg->max_tokens) return EP_ERR_INVALID_ARG;
  const bool prequant = d_x_q != nullptr || d_x_scale != nullptr;
  if (prequant && (d_x != nullptr || d_x_q == nullptr || d_x_scale == nullptr))
    return EP_ERR_INVALID_ARG;  // exactly one input form
  if (T > 0) {
    if (!prequant && (d_x == nullptr || !aligned16(d_x))) return EP_ERR_INVALID_ARG;
    if (prequant && (!aligned16(d_x_q) || !aligned16(d_x_scale))) return EP_ERR_INVALID_ARG;
  }
  if (d_recv_q == nullptr || !aligned16(d_recv_q)) return EP_ERR_INVALID_ARG;
  if (d_recv_scale == nullptr || !aligned16(d_recv_scale)) return EP_ERR_INVALID_ARG;
  if (d_topk_weights != nullptr && !aligned16(d_topk_weights)) return EP_ERR_INVALID_ARG;
  if (d_recv_w != nullptr && (!aligned16(d_recv_w) || d_topk_weights == nullptr))
    return EP_ERR_INVALID_ARG;
  if (ensure_prepared() != cudaSuccess) return EP_ERR_CUDA;
  DispatchArgs a;
  a.x = d_x;
  a.topk_weights = d_topk_weights;
  a.slot_of = layout->slot_of;
  a.expert_start = layout->expert_start;
  a.expert_end = layout->expert_end;
  a.T = T;
  a.H = cfg->hidden;
  a.K = cfg->num_topk;
  a.E = cfg->num_experts;
  a.fp8 = true;
  a.zero_padding = cfg->zero_padding != 0;
  a.recv_x = d_recv_q;
  a.recv_scale = d_recv_scale;
  a.recv_w = d_recv_w;
  a.err = layout->err;
  a.x_q = d_x_q;
  a.x_scale = d_x_scale;
  a.scale_col_major = scale_col_major != 0;
  a.scale_ld = (capacity(cfg) + 3) / 4 * 4;
  return cuda_status(launch_dispatch(a, static_cast<cudaStream_t>(stream)));
}

int32_t ep_combine_epilogue(const ep_config* cfg, const ep_layout* layout,
                            const void* d_expert_out, const float* d_topk_weights,
                            const void* d_bias0, const void* d_bias1,
                            const float* d_recv_w, void* d_y, float* d_combined_w,
                            void* stream) {
  if (!config_ok(cfg) || !layout_ptrs_ok(layout)) return EP_ERR_INVALID_ARG;
  const int T = layout->num_tokens;
  if (T < 0 || T > cfg->max_tokens) return EP_ERR_INVALID_ARG;
  if (T > 0) {
    if (d_expert_out == nullptr || !aligned16(d_expert_out)) return EP_ERR_INVALID_ARG;
    if (d_y == nullptr || !aligned16(d_y)) return EP_ERR_INVALID_ARG;
  }
  const void* ptrs[] = {d_topk_weights, d_bias0, d_bias1, d_recv_w, d_combined_w};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return EP_ERR_INVALID_ARG;
  if (d_combined_w != nullptr && d_recv_w == nullptr) return EP_ERR_INVALID_ARG;
  if (ensure_prepared() != cudaSuccess) return EP_ERR_CUDA;
  CombineArgs a;
  a.expert_out = d_expert_out;
  a.topk_weights = d_topk_weights;
  a.slot_of = layout->slot_of;
  a.T = T;
  a.H = cfg->hidden;
  a.K = cfg->num_topk;
  a.y = d_y;
  a.bias0 = d_bias0;
  a.bias1 = d_bias1;
  a.recv_w = d_recv_w;
  a.combined_w = d_combined_w;
  return cuda_status(launch_combine(a, static_cast<cudaStream_t>(stream)));
}

int32_t ep_dispatch_backward(const ep_config* cfg, const ep_layout* layout,
                             const void* d_grad_recv, const float* d_grad_recv_w,
                             void* d_grad_x, float* d_grad_w, void* stream) {
  if (!config_ok(cfg) || !layout_ptrs_ok(layout)) return EP_ERR_INVALID_ARG;
  const int T = layout->num_tokens;
  if (T < 0 || T > cfg->max_tokens) return EP_ERR_INVALID_ARG;
  if (T > 0) {
    if (d_grad_recv == nullptr || !aligned16(d_grad_recv)) return EP_ERR_INVALID_ARG;
    if (d_grad_x == nullptr || !aligned16(d_grad_x)) return EP_ERR_INVALID_ARG;
  }
  if ((d_grad_w == nullptr) != (d_grad_recv_w == nullptr)) return EP_ERR_INVALID_ARG;
  if (d_grad_w != nullptr && (!aligned16(d_grad_w) || !aligned16(d_grad_recv_w)))
    return EP_ERR_INVALID_ARG;
  if (ensure_prepared() != cudaSuccess) return EP_ERR_CUDA;
  // The transpose of the bit-copy dispatch is the unweighted row sum.
  CombineArgs a;
  a.expert_out = d_grad_recv;
  a.topk_weights = nullptr;
  a.slot_of = layout->slot_of;
  a.T = T;
  a.H = cfg->hidden;
  a.K = cfg->num_topk;
  a.y = d_grad_x;
  a.recv_w = d_grad_recv_w;
  a.combined_w = d_grad_w;
  return cuda_status(launch_combine(a, static_cast<cudaStream_t>(stream)));
}

int32_t ep_combine_backward(const ep_config* cfg, const ep_layout* layout,
                            const void* d_dy, const float* d_topk_weights,
                            const void* d_expert_out, void* d_grad_expert_out,
                            float* d_grad_w, void* stream) {
  if (!config_ok(cfg) || !layout_ptrs_ok(layout)) return EP_ERR_INVALID_ARG;
  const int T = layout->num_tokens;
  if (T < 0 || T > cfg->max_tokens) return EP_ERR_INVALID_ARG;
  if (d_grad_expert_out == nullptr || !aligned16(d_grad_expert_out)) return EP_ERR_INVALID_ARG;
  if (T > 0 && (d_dy == nullptr || !aligned16(d_dy))) return EP_ERR_INVALID_ARG;
  if (d_topk_weights != nullptr && !aligned16(d_topk_weights)) return EP_ERR_INVALID_ARG;
  if (d_grad_w != nullptr &&
      (!aligned16(d_grad_w) || d_expert_out == nullptr || !aligned16(d_expert_out)))
    return EP_ERR_INVALID_ARG;
  if (ensure_prepared() != cudaSuccess) return EP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CombineBackwardArgs a;
  a.dy = d_dy;
  a.topk_weights = d_topk_weights;
  a.slot_of = layout->slot_of;
  a.expert_out = d_expert_out;
  a.T = T;
  a.H = cfg->hidden;
  a.K = cfg->num_topk;
  a.grad_expert_out = d_grad_expert_out;
  a.grad_w = d_grad_w;
  cudaError_t e = launch_combine_backward(a, s);
  if (e == cudaSuccess && cfg->zero_padding)
    e = launch_zero_padding_bf16(layout->expert_start, layout->expert_end,
                                 cfg->num_experts, cfg->hidden, d_grad_expert_out, s);
  return cuda_status(e);
}

int64_t ep_rank_rows_capacity(const ep_config* cfg) {
  return config_ok(cfg) ? rank_rows_capacity(cfg) : -1;
}

// Common checks of the non-expanded entry points.
static int32_t rank_call_ok(const ep_config* cfg, const ep_layout* layout,
                            const void* const* required, int n_required,
                            const void* const* optional, int n_optional) {
  if (!config_ok(cfg) || !layout_ptrs_ok(layout) || !has_rank_rows(layout))
    return EP_ERR_INVALID_ARG;
  const int T = layout->num_tokens;
  if (T < 0 || T > cfg->max_tokens) return EP_ERR_INVALID_ARG;
  if (T > 0)
    for (int i = 0; i < n_required; ++i)
      if (required[i] == nullptr || !aligned16(required[i])) return EP_ERR_INVALID_ARG;
  for (int i = 0; i < n_optional; ++i)
    if (optional[i] != nullptr && !aligned16(optional[i])) return EP_ERR_INVALID_ARG;
  if (ensure_prepared() != cudaSuccess) return EP_ERR_CUDA;
  return EP_OK;
}

static RankArgs rank_args(const ep_config* cfg, const ep_layout* layout, RankArgs::Op op) {
  RankArgs a = {};
  a.op = op;
  a.slot_of = layout->slot_of;
  a.rank_slot_of = layout->rank_slot_of;
  a.T = layout->num_tokens;
  a.H = cfg->hidden;
  a.K = cfg->num_topk;
  a.E = cfg->num_experts;
  a.R = cfg->num_ranks;
  return a;
}

int32_t ep_dispatch_ranks(const ep_config* cfg, const ep_layout* layout,
                          const void* d_x, const int64_t* d_topk_idx,
                          const float* d_topk_weights, void* d_rank_x,
                          int32_t* d_rank_topk_idx, float* d_rank_topk_w,
                          void* stream) {
  const void* req[] = {d_x, d_topk_idx, d_rank_x, d_rank_topk_idx};
  const void* opt[] = {d_topk_weights, d_rank_topk_w};
  int32_t st = rank_call_ok(cfg, layout, req, 4, opt, 2);
  if (st != EP_OK) return st;
  RankArgs a = rank_args(cfg, layout, RankArgs::kDispatch);
  a.src = d_x;
  a.dst = d_rank_x;
  a.topk_idx = d_topk_idx;
  a.weights = d_topk_weights;
  a.rank_topk_idx = d_rank_topk_idx;
  a.rank_topk_w = d_rank_topk_w;
  return cuda_status(launch_ranks(a, static_cast<cudaStream_t>(stream)));
}

int32_t ep_expand(const ep_config* cfg, const ep_layout* layout,
                  const int64_t* d_topk_idx, const void* d_rank_x,
                  const float* d_rank_topk_w, void* d_recv_x, float* d_recv_w,
                  void* stream) {
  const void* req[] = {d_topk_idx, d_rank_x, d_recv_x};
  const void* opt[] = {d_rank_topk_w, d_recv_w};
  int32_t st = rank_call_ok(cfg, layout, req, 3, opt, 2);
  if (st != EP_OK) return st;
  if ((d_recv_w == nullptr) != (d_rank_topk_w == nullptr)) return EP_ERR_INVALID_ARG;
  RankArgs a = rank_args(cfg, layout, RankArgs::kExpand);
  a.src = d_rank_x;
  a.dst = d_recv_x;
  a.topk_idx = d_topk_idx;
  a.rank_topk_w = const_cast<float*>(d_rank_topk_w);
  a.recv_w = d_recv_w;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_ranks(a, s);
  if (e == cudaSuccess && cfg->zero_padding)
    e = launch_zero_padding_bf16(layout->expert_start, layout->expert_end,
                                 cfg->num_experts, cfg->hidden, d_recv_x, s);
  return cuda_status(e);
}

int32_t ep_reduce_ranks(const ep_config* cfg, const ep_layout* layout,
                        const int64_t* d_topk_idx, const void* d_expert_out,
                        const float* d_topk_weights, void* d_rank_y, void* stream) {
  const void* req[] = {d_topk_idx, d_expert_out, d_rank_y};
  const void* opt[] = {d_topk_weights};
  int32_t st = rank_call_ok(cfg, layout, req, 3, opt, 1);
  if (st != EP_OK) return st;
  RankArgs a = rank_args(cfg, layout, RankArgs::kReduce);
  a.src = d_expert_out;
  a.dst = d_rank_y;
  a.topk_idx = d_topk_idx;
  a.weights = d_topk_weights;
  return cuda_status(launch_ranks(a, static_cast<cudaStream_t>(stream)));
}

int32_t ep_combine_ranks(const ep_config* cfg, const ep_layout* layout,
                         const void* d_rank_y, void* d_y, void* stream) {
  const void* req[] = {d_rank_y, d_y};
  int32_t st = rank_call_ok(cfg, layout, req, 2, nullptr, 0);
  if (st != EP_OK) return st;
  if (cfg->num_ranks > kCombineMaxSlots) return EP_ERR_INVALID_ARG;
  // The unweighted row sum over the token's rank rows, in ascending rank.
  CombineArgs a;
  a.expert_out = d_rank_y;
  a.topk_weights = nullptr;
  a.slot_of = layout->rank_slot_of;
  a.T = layout->num_tokens;
  a.H = cfg->hidden;
  a.K = cfg->num_ranks;
  a.y = d_y;
  return cuda_status(launch_combine(a, static_cast<cudaStream_t>(stream)));
}

int32_t ep_check_error(const ep_layout* layout, void* stream) {
  if (layout == nullptr || layout->err == nullptr) return EP_ERR_INVALID_ARG;
  int32_t bits = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&bits, layout->err, sizeof(int32_t),
                                  cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (note_cuda(e) != cudaSuccess) return EP_ERR_CUDA;
  return status_from_bits(bits);
}

int32_t ep_selftest_fp8_quotient(uint64_t* d_counts, int32_t* d_first, void* stream) {
  if (d_counts == nullptr || d_first == nullptr || !aligned16(d_counts))
    return EP_ERR_INVALID_ARG;
  if (ensure_prepared() != cudaSuccess) return EP_ERR_CUDA;
  return cuda_status(launch_fp8_quotient_selftest(
      reinterpret_cast<unsigned long long*>(d_counts), d_first,
      static_cast<cudaStream_t>(stream)));
}

int32_t ep_selftest_wait_timeout(int64_t timeout_ns, int32_t* d_err, void* stream) {
  if (d_err == nullptr || !aligned16(d_err)) return EP_ERR_INVALID_ARG;
  if (timeout_ns < 1000 || timeout_ns > 1000000000) return EP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_wait_selftest(uint64_t(timeout_ns), d_err, s);
  int32_t bits = 0;
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&bits, d_err, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (note_cuda(e) != cudaSuccess) return EP_ERR_CUDA;
  return status_from_bits(bits);
}

int32_t ep_selftest_layout_timeout(const ep_config* cfg, int32_t num_tokens,
                                   const int64_t* d_topk_idx, ep_layout* layout,
                                   int32_t stall_tile, int64_t timeout_ns, void* stream) {
  LayoutArgs a;
  const int32_t v = layout_args(cfg, num_tokens, d_topk_idx, layout, &a);
  if (v != EP_OK) return v;
  if (timeout_ns < 1000 || timeout_ns > 1000000000) return EP_ERR_INVALID_ARG;
  // the two-launch layout only (the one-launch layout has no waits)
  if (num_tokens == 0 || layout_is_small(num_tokens, a.K, a.E)) return EP_ERR_INVALID_ARG;
  if (stall_tile < 0 || stall_tile >= assign_grid(a.geom.num_tiles, a.E))
    return EP_ERR_INVALID_ARG;
  if (ensure_prepared() != cudaSuccess) return EP_ERR_CUDA;
  a.stall_tile = stall_tile;
  a.wait_ns = uint64_t(timeout_ns);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_layout(a, s);
  layout->num_tokens = num_tokens;
  int32_t bits = 0;
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&bits, layout->err, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (note_cuda(e) != cudaSuccess) return EP_ERR_CUDA;
  return status_from_bits(bits);
}

int32_t ep_last_cuda_error(void) {
  const cudaError_t e = g_last_cuda_error;
  g_last_cuda_error = cudaSuccess;
  return static_cast<int32_t>(e);
}

const char* ep_status_str(int32_t status) {
  switch (status) {
    case EP_OK: return "EP_OK";
    case EP_ERR_INVALID_ARG: return "EP_ERR_INVALID_ARG";
    case EP_ERR_EXPERT_RANGE: return "EP_ERR_EXPERT_RANGE";
    case EP_ERR_DUP_EXPERT: return "EP_ERR_DUP_EXPERT";
    case EP_ERR_CAPACITY: return "EP_ERR_CAPACITY";
    case EP_ERR_CUDA: return "EP_ERR_CUDA";
    case EP_ERR_TIMEOUT: return "EP_ERR_TIMEOUT";
    case EP_ERR_TIMEOUT_PENDING: return "EP_ERR_TIMEOUT_PENDING";
    default: return "EP_ERR_UNKNOWN";
  }
}

}  // extern "C"

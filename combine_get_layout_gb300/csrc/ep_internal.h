// Host-side declarations shared by the translation units of libep_gb300.so:
// kernel launchers (defined next to their kernels) and launch geometry.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace ep {

// Layout tiling: a tile is a run of whole tokens handled by one CTA of
// kLayoutThreads threads.  There are at most kLayoutMaxTiles tiles, each of
// at least kMinTilePairs (t, k) pairs when the input allows.
constexpr int kLayoutThreads = 256;
constexpr int kLayoutWarps = kLayoutThreads / 32;
// Threads of an assign-kernel CTA.  (1024, with the extra warps on the
// column sums, scans and stores only, measured slower at 4K-16K tokens: the
// larger CTAs start later.)
constexpr int kAssignThreads = kLayoutThreads;
constexpr int kLayoutMaxTiles = 152;
constexpr int kMinTilePairs = 256;
// The assign kernel loads the whole tile-count matrix with one bulk copy
// when it fits, with the kernel's other shared arrays, in kAssignSmemBudget
// bytes; otherwise it streams it through two buffers of about
// kScanChunkBytes.
constexpr int kAssignSmemBudget = 220 * 1024;
constexpr int kScanChunkBytes = 32 * 1024;
// Inputs of at most kSmallLayoutPairs (t, k) pairs, with at most
// kSmallLayoutMaxExperts experts, take the one-launch layout.
constexpr int kSmallLayoutPairs = 4096;
constexpr int kSmallLayoutMaxExperts = 2048;
// Threads of a one-launch layout CTA: a pair a thread at decode sizes, and
// warps enough to hide the latency of its short dependent phases.
constexpr int kSmallThreads = 1024;
constexpr int kSmallWarps = kSmallThreads / 32;
bool layout_is_small(int64_t T, int K, int E);
// Pairs a CTA of the one-launch layout may own when it also dispatches them.
constexpr int kSmallOwnPairs = 64;
// Shared memory up to which the one-launch layout also stages the x rows of
// its own tokens when it dispatches them.
constexpr int kSmallStageBudget = 200 * 1024;


struct TileGeom {
  int tile_tokens;  // tokens per tile (last tile may be short)
  int num_tiles;
};

// Geometry for T tokens of K selections each (T >= 1).
TileGeom layout_tiles(int64_t T, int K);

// Experts padded to a multiple of 4 (rows of the tile-count matrix are then
// 16-byte multiples, as bulk copies need).
__host__ __device__ inline int padded_experts(int E) { return (E + 3) & ~3; }

// Ranks padded to a multiple of 4 likewise.
__host__ __device__ inline int padded_ranks(int R) { return (R + 3) & ~3; }
// Width of a tile-count row: expert counts then rank counts.
__host__ __device__ inline int count_row_width(int E, int R) {
  return padded_experts(E) + padded_ranks(R);
}

// Entries of a tile-count row as the count kernel stores it: 32-bit
// counts, or 16-bit counts (when a tile holds at most 65535 (t, k) pairs)
// with the row rounded up to 8 entries so that it stays a 16-byte multiple.
__host__ __device__ inline int count_row_entries(int E, int R, bool k16) {
  const int Wc = count_row_width(E, R);
  return k16 ? (Wc + 7) & ~7 : Wc;
}
__host__ __device__ inline int count_row_bytes(int E, int R, bool k16) {
  return count_row_entries(E, R, k16) * (k16 ? 2 : 4);
}

// Workspace carved by ep_get_layout (arrays 16-byte aligned):
//   tile_counts: kLayoutMaxTiles rows of count_row_bytes (row c: tile c's
//   expert counts, then its rank counts; sized for 32-bit counts, the
//   16-bit form uses part of it), tile_err [kLayoutMaxTiles] int32.
struct LayoutWorkspace {
  int32_t* tile_counts;
  int32_t* tile_err;
};
int64_t layout_workspace_bytes(int E, int R);
LayoutWorkspace carve_layout_workspace(void* base, int E, int R);

struct LayoutArgs {
  const int64_t* topk_idx;
  int T, K, E, R, A;
  TileGeom geom;
  LayoutWorkspace ws;
  int32_t *expert_count, *expert_start, *expert_end, *rank_start;
  int32_t *tokens_per_rank, *slot_of, *src_info, *err;
  uint8_t* is_token_in_rank;
  // optional rank rows (all set or all null)
  int32_t *rank_row_start = nullptr, *rank_slot_of = nullptr, *rank_src = nullptr;
  // self-test of the assign kernel's bounded wait: the CTA numbered
  // stall_tile issues no copy and waits wait_ns for it (-1: none)
  int stall_tile = -1;
  uint64_t wait_ns = 1000ull * 1000ull * 1000ull;
};

cudaError_t launch_layout(const LayoutArgs& a, cudaStream_t stream);

// CTAs of the assign kernel for a layout of `tiles` tiles over E experts.
int assign_grid(int tiles, int E);

// Dispatch work handed to the one-launch layout (layout_small_kernel).
struct SmallDispatch {
  const uint4* x = nullptr;       // bf16 [T, H]
  const float* w = nullptr;       // [T, K] or null
  void* recv_x = nullptr;         // bf16 or E4M3 rows
  float* recv_scale = nullptr;    // [cap, H/128] row-major (E4M3)
  float* recv_w = nullptr;        // [cap] or null
  int H = 0;
};

struct DispatchArgs {
  const void* x;
  const float* topk_weights;
  const int32_t* slot_of;
  const int32_t* expert_start;
  const int32_t* expert_end;
  int T, H, K, E;
  bool fp8;
  bool zero_padding;
  void* recv_x;
  float* recv_scale;
  float* recv_w;
  int32_t* err;
  // FP8 options: pre-quantised input (E4M3 rows + fp32 scales) instead of
  // x, and column-major scales with leading dimension scale_ld.
  const uint8_t* x_q = nullptr;
  const float* x_scale = nullptr;
  // programmatic dependent launch of the row kernels (off after a wait on
  // another stream)
  bool pdl = true;
  bool scale_col_major = false;
  int64_t scale_ld = 0;
};

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t stream);

struct CombineArgs {
  const void* expert_out;
  const float* topk_weights;
  const int32_t* slot_of;
  int T, H, K;
  void* y;
  // epilogue (all optional)
  const void* bias0 = nullptr;
  const void* bias1 = nullptr;
  const float* recv_w = nullptr;
  float* combined_w = nullptr;
  bool pdl = true;   // as in DispatchArgs
};

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream);

struct CombineBackwardArgs {
  const void* dy;                 // bf16 [T, H]
  const float* topk_weights;      // [T, K] or null (weight 1)
  const int32_t* slot_of;
  const void* expert_out;         // bf16 [cap, H]; needed when grad_w is set
  int T, H, K;
  void* grad_expert_out;          // bf16 [cap, H]
  float* grad_w;                  // [T, K] or null
};

cudaError_t launch_combine_backward(const CombineBackwardArgs& a, cudaStream_t stream);

// Zeroes the alignment gap rows of a bf16 [cap, H] buffer (rows
// [expert_end[e], expert_start[e+1])).
cudaError_t launch_zero_padding_bf16(const int32_t* expert_start, const int32_t* expert_end,
                                     int E, int H, void* rows, cudaStream_t stream);

// Non-expanded stage kernels (csrc/ranks.cu).
struct RankArgs {
  enum Op { kDispatch, kExpand, kReduce } op;
  const void* src;              // x (dispatch), rank_x (expand), expert rows (reduce)
  void* dst;                    // rank_x (dispatch), recv_x (expand), rank_y (reduce)
  const int64_t* topk_idx;
  const float* weights;         // topk_weights (dispatch, reduce) or null
  const int32_t* slot_of;
  const int32_t* rank_slot_of;
  int32_t* rank_topk_idx;       // dispatch output
  float* rank_topk_w;           // dispatch output / expand input (optional)
  float* recv_w;                // expand output (optional)
  int T, H, K, E, R;
};

cudaError_t launch_ranks(const RankArgs& a, cudaStream_t stream);

// Layout then dispatch; for small inputs one launch does both (the CTAs of
// the one-launch layout dispatch their own tokens), else the two paths run
// in turn.  Results equal launch_layout followed by launch_dispatch.
cudaError_t launch_layout_dispatch(const LayoutArgs& la, const DispatchArgs& da,
                                   cudaStream_t stream);

// Threads per CTA and CTAs per token (grid.y) for a row of nvec vectors: the
// fewest CTAs of at most `cap` threads, balanced, in whole warps.  Several
// CTAs per token let one CTA's short per-token preamble overlap another's
// stream on the same SM.
inline void split_row(int nvec, int cap, dim3* block, int* parts) {
  const int p = nvec > 0 ? (nvec + cap - 1) / cap : 1;
  const int per = (nvec + p - 1) / p;
  *block = dim3(((per + 31) / 32) * 32);
  *parts = p;
}

// Largest K the combine kernel reads per token (top-k selections, or rank
// rows when it sums over destination ranks).
constexpr int kCombineMaxSlots = 64;

// Exhaustive check of the FP8 dispatch's quotient against the IEEE division
// (counts[3]: E4M3 code mismatches, fp32 mismatches, fp32 mismatches with
// a normal IEEE quotient; first: one code mismatch or -1).
cudaError_t launch_fp8_quotient_selftest(unsigned long long* counts, int32_t* first,
                                         cudaStream_t stream);

// One CTA waiting (bounded) on a barrier nothing completes.
cudaError_t launch_wait_selftest(uint64_t timeout_ns, int32_t* err, cudaStream_t stream);

// Launches `kernel` with programmatic stream serialisation (see pdl_wait in
// ep_device.cuh).
// With pdl = false the launch is an ordinary stream-ordered one (used after
// a wait on another stream's event, where the kernel must not start early).
template <typename... Params, typename... Args>
cudaError_t launch_ex(bool pdl, void (*kernel)(Params...), dim3 grid, dim3 block,
                      size_t smem, cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block,
                       size_t smem, cudaStream_t stream, Args&&... args) {
  return launch_ex(true, kernel, grid, block, smem, stream, std::forward<Args>(args)...);
}

// Raises `kernel`'s dynamic shared-memory limit to what the device allows
// next to the kernel's static shared memory.
template <typename... Params>
cudaError_t allow_max_dynamic_smem(void (*kernel)(Params...), int optin) {
  cudaFuncAttributes fa;
  cudaError_t st = cudaFuncGetAttributes(&fa, kernel);
  if (st != cudaSuccess) return st;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              optin - static_cast<int>(fa.sharedSizeBytes));
}

// Records a failed CUDA runtime status for ep_last_cuda_error (per thread).
cudaError_t note_cuda(cudaError_t e);

// Per-device one-time set-up of the kernels' shared-memory limits.
cudaError_t prepare_layout_kernels();
cudaError_t prepare_dispatch_kernels();

// Cached per-device properties (queried once per device).
struct DeviceInfo {
  int sm_count;
  int max_smem_optin;   // bytes of shared memory a CTA may opt into
  int smem_per_sm;      // bytes of shared memory per SM
};
const DeviceInfo& device_info();

}  // namespace ep

// Host-side declarations shared by the translation units of libep_gb300.so:
// kernel launchers (defined next to their kernels) and launch geometry.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ep {

// Layout tiling: a tile is a run of whole tokens handled by one CTA of
// kLayoutThreads threads.  Tiles are sized so that about kLayoutTargetTiles
// CTAs run, each with between kMinTilePairs and kMaxTilePairs (t, k) pairs.
constexpr int kLayoutThreads = 256;
constexpr int kLayoutWarps = kLayoutThreads / 32;
constexpr int kLayoutTargetTiles = 152;
constexpr int kMinTilePairs = 256;
constexpr int kMaxTilePairs = 4096;

struct TileGeom {
  int tile_tokens;  // tokens per tile (last tile may be short)
  int num_tiles;
};

// Geometry for T tokens of K selections each (T >= 1).
TileGeom layout_tiles(int64_t T, int K);
// Largest tile count any T <= max_tokens can produce.
int layout_max_tiles(int64_t max_tokens, int K);

// Workspace carved by ep_get_layout (int32 arrays, each 16-byte aligned):
//   tile_counts [tiles * E], tile_base [tiles * E],
//   tile_rank_counts [tiles * R], tile_err [tiles].
struct LayoutWorkspace {
  int32_t* tile_counts;
  int32_t* tile_base;
  int32_t* tile_rank_counts;
  int32_t* tile_err;
};
int64_t layout_workspace_bytes(int max_tiles, int E, int R);
LayoutWorkspace carve_layout_workspace(void* base, int max_tiles, int E, int R);

struct LayoutArgs {
  const int64_t* topk_idx;
  int T, K, E, R, A;
  TileGeom geom;
  LayoutWorkspace ws;
  int32_t *expert_count, *expert_start, *expert_end, *rank_start;
  int32_t *tokens_per_rank, *slot_of, *src_info, *err;
  uint8_t* is_token_in_rank;
};

cudaError_t launch_layout(const LayoutArgs& a, cudaStream_t stream);

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
};

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t stream);

struct CombineArgs {
  const void* expert_out;
  const float* topk_weights;
  const int32_t* slot_of;
  int T, H, K;
  void* y;
};

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream);

// One CTA waiting (bounded) on a barrier nothing completes.
cudaError_t launch_wait_selftest(uint64_t timeout_ns, int32_t* err, cudaStream_t stream);

// Cached per-device properties (queried once per device).
struct DeviceInfo {
  int sm_count;
  int max_smem_optin;   // bytes of shared memory a CTA may opt into
  int smem_per_sm;      // bytes of shared memory per SM
};
const DeviceInfo& device_info();

}  // namespace ep

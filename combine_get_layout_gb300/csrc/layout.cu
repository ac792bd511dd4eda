// Layout kernels: count -> prefix sum -> scatter ("GPU Microarchitecture:
// DeepEP from First Principles", 6.1 Layout Metadata and 7.1 Does Sort
// Exist?), with the expanded-mode alignment and psum semantics of "Deep Dive
// - DeepEP", "Dispatch: layout, move, and epilogue", and rows ordered by
// source-global order ("EPHandle: route metadata with a lifetime").
//
// Three launches, no inter-CTA waiting:
//   1. count   (one CTA per token tile): validate topk_idx, per-tile expert
//      histogram with warp-aggregated shared-memory atomics, per-rank dedup
//      flags and per-tile rank counts.
//   2. scan    (one CTA): per expert, exclusive scan of the tile counts over
//      tiles; per-expert totals; aligned exclusive scan over experts;
//      rank ranges, tokens per rank, error word.
//   3. assign  (one CTA per tile): recount per warp, turn the counts into
//      per-warp bases, and give each (t, k) its row.  Warps own contiguous
//      runs of (t, k) pairs and walk them in order, so rows within an expert
//      follow (t, k) order whatever the scheduling.
#include "ep_device.cuh"
#include "ep_internal.h"

namespace ep {

TileGeom layout_tiles(int64_t T, int K) {
  int64_t pairs = T * K;
  int64_t target = (pairs + kLayoutTargetTiles - 1) / kLayoutTargetTiles;
  if (target < kMinTilePairs) target = kMinTilePairs;
  if (target > kMaxTilePairs) target = kMaxTilePairs;
  int64_t tt = (target + K - 1) / K;
  const int64_t max_tt = kMaxTilePairs / K;
  if (tt > max_tt) tt = max_tt;
  if (tt < 1) tt = 1;
  TileGeom g;
  g.tile_tokens = static_cast<int>(tt);
  g.num_tiles = static_cast<int>((T + tt - 1) / tt);
  return g;
}

int layout_max_tiles(int64_t max_tokens, int K) {
  if (max_tokens < 1) return 1;
  int64_t m = kLayoutTargetTiles + 2;
  int64_t big = (max_tokens + (kMaxTilePairs / K) - 1) / (kMaxTilePairs / K);
  if (big > m) m = big;
  int64_t at_max = layout_tiles(max_tokens, K).num_tiles;
  if (at_max > m) m = at_max;
  return static_cast<int>(m);
}

static int64_t round16(int64_t b) { return (b + 15) & ~int64_t(15); }

int64_t layout_workspace_bytes(int max_tiles, int E, int R) {
  return 2 * round16(int64_t(max_tiles) * E * 4) +
         round16(int64_t(max_tiles) * R * 4) + round16(int64_t(max_tiles) * 4);
}

LayoutWorkspace carve_layout_workspace(void* base, int max_tiles, int E, int R) {
  char* p = static_cast<char*>(base);
  LayoutWorkspace ws;
  ws.tile_counts = reinterpret_cast<int32_t*>(p);
  p += round16(int64_t(max_tiles) * E * 4);
  ws.tile_base = reinterpret_cast<int32_t*>(p);
  p += round16(int64_t(max_tiles) * E * 4);
  ws.tile_rank_counts = reinterpret_cast<int32_t*>(p);
  p += round16(int64_t(max_tiles) * R * 4);
  ws.tile_err = reinterpret_cast<int32_t*>(p);
  return ws;
}

// Loads one tile of topk_idx into shared memory as int32, validating it:
// an id outside [-1, E) is recorded and treated as unused (-1) from here on,
// so that no later kernel can index out of range.
__device__ __forceinline__ int load_tile_idx(const int64_t* __restrict__ src,
                                             int P, int E,
                                             int32_t* __restrict__ sidx) {
  int err = 0;
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int64_t v = src[p];
    int32_t e = static_cast<int32_t>(v);
    if (v < -1 || v >= E) {
      err |= ERRBIT_EXPERT_RANGE;
      e = -1;
    }
    sidx[p] = e;
  }
  return err;
}

// ---------------------------------------------------------------------------
// 1. count
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kLayoutThreads)
    layout_count_kernel(const int64_t* __restrict__ topk_idx, int T, int K,
                        int E, int R, int tile_tokens,
                        int32_t* __restrict__ tile_counts,
                        int32_t* __restrict__ tile_rank_counts,
                        int32_t* __restrict__ tile_err,
                        uint8_t* __restrict__ is_token_in_rank) {
  extern __shared__ int32_t smem_i32[];
  __shared__ int32_t s_err;
  const int tile = blockIdx.x;
  const int t0 = tile * tile_tokens;
  const int nt = min(tile_tokens, T - t0);
  const int P = nt * K;
  int32_t* sidx = smem_i32;
  int32_t* hist = sidx + tile_tokens * K;
  int32_t* rcnt = hist + E;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) s_err = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  for (int r = threadIdx.x; r < R; r += blockDim.x) rcnt[r] = 0;
  int err = load_tile_idx(topk_idx + int64_t(t0) * K, P, E, sidx);
  __syncthreads();

  // Expert histogram.  Lanes holding the same expert are grouped with
  // match.any; only the group's first lane touches shared memory, so a hot
  // expert (skewed routing) costs one atomic per warp, not one per lane.
  for (int base = 0; base < P; base += blockDim.x) {
    const int p = base + threadIdx.x;
    const int e = p < P ? sidx[p] : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[e], __popc(peers));
  }

  // An expert may appear once per token (-1 may repeat).
  for (int t = threadIdx.x; t < nt; t += blockDim.x) {
    const int32_t* row = sidx + t * K;
    for (int k = 0; k < K; ++k)
      for (int k2 = k + 1; k2 < K; ++k2)
        if (row[k] >= 0 && row[k] == row[k2]) err |= ERRBIT_DUP_EXPERT;
  }

  // Destination ranks: a token goes once to every rank owning one of its
  // experts (owner rank = expert / experts-per-rank).
  const int Eg = E / R;
  for (int i = threadIdx.x; i < nt * R; i += blockDim.x) {
    const int t = i / R;
    const int r = i - t * R;
    const int32_t* row = sidx + t * K;
    int in = 0;
    for (int k = 0; k < K; ++k) in |= (row[k] >= 0) & (row[k] / Eg == r);
    is_token_in_rank[int64_t(t0) * R + i] = static_cast<uint8_t>(in);
    if (in) atomicAdd(&rcnt[r], 1);
  }
  if (err) atomicOr(&s_err, err);
  __syncthreads();

  for (int e = threadIdx.x; e < E; e += blockDim.x)
    tile_counts[int64_t(tile) * E + e] = hist[e];
  for (int r = threadIdx.x; r < R; r += blockDim.x)
    tile_rank_counts[int64_t(tile) * R + r] = rcnt[r];
  if (threadIdx.x == 0) tile_err[tile] = s_err;
}

// ---------------------------------------------------------------------------
// 2. scan (single CTA of kScanThreads threads)
// ---------------------------------------------------------------------------
constexpr int kScanThreads = 1024;

// Block-wide exclusive scan of one int per thread; returns the exclusive
// prefix and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int32_t* s_warp,
                                                    int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;  // inclusive prefix over warps
  }
  __syncthreads();
  const int warp_excl = warp > 0 ? s_warp[warp - 1] : 0;
  *total = s_warp[(blockDim.x >> 5) - 1];
  __syncthreads();
  return warp_excl + x - v;
}

__global__ void __launch_bounds__(kScanThreads)
    layout_scan_kernel(int num_tiles, int E, int R, int A,
                       const int32_t* __restrict__ tile_counts,
                       int32_t* __restrict__ tile_base,
                       const int32_t* __restrict__ tile_rank_counts,
                       const int32_t* __restrict__ tile_err,
                       int32_t* __restrict__ expert_count,
                       int32_t* __restrict__ expert_start,
                       int32_t* __restrict__ expert_end,
                       int32_t* __restrict__ rank_start,
                       int32_t* __restrict__ tokens_per_rank,
                       int32_t* __restrict__ err) {
  extern __shared__ int32_t smem_i32[];
  __shared__ int32_t s_warp[32];
  __shared__ int32_t s_err;
  const int tid = threadIdx.x;
  if (tid == 0) s_err = 0;

  // (a) per expert: exclusive scan over tiles.  G groups of threads split
  // the tiles into contiguous ranges so that each thread has few loads.
  int G = kScanThreads / E;
  if (G < 1) G = 1;
  if (G > 32) G = 32;
  const int per = (num_tiles + G - 1) / G;
  int32_t* part = smem_i32;  // [G * E]
  for (int i = tid; i < G * E; i += kScanThreads) {
    const int g = i / E, e = i - g * E;
    const int c0 = g * per, c1 = min(num_tiles, c0 + per);
    int s = 0;
#pragma unroll 8
    for (int c = c0; c < c1; ++c) s += tile_counts[int64_t(c) * E + e];
    part[i] = s;
  }
  __syncthreads();
  for (int e = tid; e < E; e += kScanThreads) {
    int run = 0;
    for (int g = 0; g < G; ++g) {
      const int v = part[g * E + e];
      part[g * E + e] = run;
      run += v;
    }
    expert_count[e] = run;
  }
  __syncthreads();
  for (int i = tid; i < G * E; i += kScanThreads) {
    const int g = i / E, e = i - g * E;
    const int c0 = g * per, c1 = min(num_tiles, c0 + per);
    int run = part[i];
#pragma unroll 8
    for (int c = c0; c < c1; ++c) {
      const int v = tile_counts[int64_t(c) * E + e];
      tile_base[int64_t(c) * E + e] = run;
      run += v;
    }
  }
  __syncthreads();

  // (b) aligned exclusive scan over experts: every segment rounded up to a
  // multiple of A; expert_end = aligned start + real count.
  const int per_t = (E + kScanThreads - 1) / kScanThreads;
  const int e0 = tid * per_t, e1 = min(E, e0 + per_t);
  int local = 0;
  for (int e = e0; e < e1; ++e) local += (expert_count[e] + A - 1) / A * A;
  int total = 0;
  int run = block_exclusive_scan(local, s_warp, &total);
  for (int e = e0; e < e1; ++e) {
    const int c = expert_count[e];
    expert_start[e] = run;
    expert_end[e] = run + c;
    run += (c + A - 1) / A * A;
  }
  if (tid == 0) expert_start[E] = total;
  __syncthreads();

  // (c) logical rank ranges and tokens per rank; the error word.
  const int Eg = E / R;
  for (int r = tid; r <= R; r += kScanThreads)
    rank_start[r] = r < R ? expert_start[r * Eg] : total;
  int Gr = kScanThreads / R;
  if (Gr < 1) Gr = 1;
  int32_t* rpart = smem_i32;  // reuse: [Gr * R]
  for (int i = tid; i < Gr * R; i += kScanThreads) {
    const int g = i / R, r = i - g * R;
    int s = 0;
    for (int c = g; c < num_tiles; c += Gr) s += tile_rank_counts[int64_t(c) * R + r];
    rpart[i] = s;
  }
  int e_or = 0;
  for (int c = tid; c < num_tiles; c += kScanThreads) e_or |= tile_err[c];
  if (e_or) atomicOr(&s_err, e_or);
  __syncthreads();
  for (int r = tid; r < R; r += kScanThreads) {
    int s = 0;
    for (int g = 0; g < Gr; ++g) s += rpart[g * R + r];
    tokens_per_rank[r] = s;
  }
  if (tid == 0) *err = s_err;
}

// ---------------------------------------------------------------------------
// 3. assign
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kLayoutThreads)
    layout_assign_kernel(const int64_t* __restrict__ topk_idx, int T, int K,
                         int E, int tile_tokens, int num_tiles,
                         const int32_t* __restrict__ tile_base,
                         const int32_t* __restrict__ expert_start,
                         const int32_t* __restrict__ expert_end,
                         int32_t* __restrict__ slot_of,
                         int32_t* __restrict__ src_info) {
  extern __shared__ int32_t smem_i32[];
  const int tile = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int2* src_info2 = reinterpret_cast<int2*>(src_info);

  if (tile < num_tiles) {
    const int t0 = tile * tile_tokens;
    const int nt = min(tile_tokens, T - t0);
    const int P = nt * K;
    int32_t* sidx = smem_i32;
    int32_t* whist = sidx + tile_tokens * K;  // [kLayoutWarps * E]
    (void)load_tile_idx(topk_idx + int64_t(t0) * K, P, E, sidx);
    for (int i = threadIdx.x; i < kLayoutWarps * E; i += blockDim.x) whist[i] = 0;
    __syncthreads();

    // Each warp owns the contiguous pairs [pb, pe) of the tile.
    const int span = (P + kLayoutWarps - 1) / kLayoutWarps;
    const int pb = min(P, warp * span), pe = min(P, pb + span);
    int32_t* my = whist + warp * E;

    for (int base = pb; base < pe; base += 32) {
      const int p = base + lane;
      const int e = p < pe ? sidx[p] : -1;
      const uint32_t peers = __match_any_sync(0xffffffffu, e);
      if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
    }
    __syncthreads();

    // Per-warp bases: aligned expert start + rows of earlier tiles + rows of
    // earlier warps of this tile.
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int run = expert_start[e] + tile_base[int64_t(tile) * E + e];
      for (int w = 0; w < kLayoutWarps; ++w) {
        const int c = whist[w * E + e];
        whist[w * E + e] = run;
        run += c;
      }
    }
    __syncthreads();

    const uint32_t lt = lanemask_lt();
    for (int base = pb; base < pe; base += 32) {
      const int p = base + lane;
      const bool in = p < pe;
      const int e = in ? sidx[p] : -1;
      const uint32_t peers = __match_any_sync(0xffffffffu, e);
      int slot = -1;
      if (e >= 0) slot = my[e] + __popc(peers & lt);
      __syncwarp();
      if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
      __syncwarp();
      if (in) {
        const int64_t gp = int64_t(t0) * K + p;
        slot_of[gp] = slot;
        if (slot >= 0) {
          const int tl = p / K;
          src_info2[slot] = make_int2(t0 + tl, p - tl * K);
        }
      }
    }
  }

  // Alignment padding rows carry no token.
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    const int s0 = expert_end[e], s1 = expert_start[e + 1];
    for (int s = s0 + threadIdx.x; s < s1; s += blockDim.x)
      src_info2[s] = make_int2(-1, -1);
  }
}

static int smem_count(int tile_tokens, int K, int E, int R) {
  return (tile_tokens * K + E + R) * 4;
}
static int smem_assign(int tile_tokens, int K, int E) {
  return (tile_tokens * K + kLayoutWarps * E) * 4;
}
static int smem_scan(int E, int R) {
  int G = kScanThreads / E;
  if (G < 1) G = 1;
  if (G > 32) G = 32;
  int Gr = kScanThreads / R;
  if (Gr < 1) Gr = 1;
  int a = G * E, b = Gr * R;
  return (a > b ? a : b) * 4;
}

cudaError_t launch_layout(const LayoutArgs& a, cudaStream_t stream) {
  const int tiles = a.T > 0 ? a.geom.num_tiles : 0;
  const int tt = a.geom.tile_tokens;
  cudaError_t st;
  if (tiles > 0) {
    const int sm = smem_count(tt, a.K, a.E, a.R);
    st = cudaFuncSetAttribute(layout_count_kernel,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    if (st != cudaSuccess) return st;
    layout_count_kernel<<<tiles, kLayoutThreads, sm, stream>>>(
        a.topk_idx, a.T, a.K, a.E, a.R, tt, a.ws.tile_counts,
        a.ws.tile_rank_counts, a.ws.tile_err, a.is_token_in_rank);
    st = cudaGetLastError();
    if (st != cudaSuccess) return st;
  }
  {
    const int sm = smem_scan(a.E, a.R);
    st = cudaFuncSetAttribute(layout_scan_kernel,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    if (st != cudaSuccess) return st;
    layout_scan_kernel<<<1, kScanThreads, sm, stream>>>(
        tiles, a.E, a.R, a.A, a.ws.tile_counts, a.ws.tile_base,
        a.ws.tile_rank_counts, a.ws.tile_err, a.expert_count, a.expert_start,
        a.expert_end, a.rank_start, a.tokens_per_rank, a.err);
    st = cudaGetLastError();
    if (st != cudaSuccess) return st;
  }
  if (tiles > 0) {
    const int sm = smem_assign(tt, a.K, a.E);
    st = cudaFuncSetAttribute(layout_assign_kernel,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    if (st != cudaSuccess) return st;
    int grid = tiles;
    const int pad_blocks = a.E < kLayoutTargetTiles ? a.E : kLayoutTargetTiles;
    if (grid < pad_blocks) grid = pad_blocks;
    layout_assign_kernel<<<grid, kLayoutThreads, sm, stream>>>(
        a.topk_idx, a.T, a.K, a.E, tt, tiles, a.ws.tile_base, a.expert_start,
        a.expert_end, a.slot_of, a.src_info);
    st = cudaGetLastError();
    if (st != cudaSuccess) return st;
  }
  return cudaSuccess;
}

}  // namespace ep

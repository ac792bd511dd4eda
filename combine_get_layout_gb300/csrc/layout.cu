// Layout kernels: count -> prefix sum -> scatter ("GPU Microarchitecture:
// DeepEP from First Principles", 6.1 Layout Metadata and 7.1 Does Sort
// Exist?), with the expanded-mode alignment and psum semantics of "Deep Dive
// - DeepEP", "Dispatch: layout, move, and epilogue", and rows ordered by
// source-global order ("EPHandle: route metadata with a lifetime").
//
// Small inputs (T * K <= kSmallLayoutPairs): one launch in which every CTA
// surveys the whole input (layout_small_kernel below).  Otherwise two
// launches, no inter-CTA waiting:
//   1. count  (one CTA per token tile): validate topk_idx, per-tile expert
//      histogram with shared-memory adds, per-rank dedup flags (a token's
//      selections compared across lanes by shuffles) and per-tile rank
//      counts.
//   2. assign (one CTA per tile, plus CTAs for padding when there are few
//      tiles): every CTA streams the whole tile-count matrix into shared
//      memory with bulk copies (TMA) and scans it itself -- its own tile
//      bases and the per-expert totals -- so there is no serial single-CTA
//      scan between the two launches.  Then the aligned exclusive scan over
//      experts, per-warp bases, and each (t, k) gets its row.  Warps own
//      contiguous runs of (t, k) pairs and walk them in order, so the rows
//      of an expert follow (t, k) order whatever the scheduling.  CTA 0
//      publishes the per-expert arrays; rank totals are spread over CTAs.
#include "ep_device.cuh"
#include "ep_internal.h"
#include "fp8_quant.cuh"

namespace ep {

TileGeom layout_tiles(int64_t T, int K) {
  const int64_t pairs = T * K;
  int64_t C = (pairs + kMinTilePairs - 1) / kMinTilePairs;
  if (C > kLayoutMaxTiles) C = kLayoutMaxTiles;
  if (C < 1) C = 1;
  int64_t tt = (T + C - 1) / C;
  if (tt < 1) tt = 1;
  TileGeom g;
  g.tile_tokens = static_cast<int>(tt);
  g.num_tiles = static_cast<int>((T + tt - 1) / tt);
  if (g.num_tiles < 1) g.num_tiles = 1;
  return g;
}

static int64_t round16(int64_t b) { return (b + 15) & ~int64_t(15); }

int64_t layout_workspace_bytes(int E, int R) {
  return round16(int64_t(kLayoutMaxTiles) * count_row_width(E, R) * 4) +
         round16(int64_t(kLayoutMaxTiles) * 4);
}

LayoutWorkspace carve_layout_workspace(void* base, int E, int R) {
  char* p = static_cast<char*>(base);
  LayoutWorkspace ws;
  ws.tile_counts = reinterpret_cast<int32_t*>(p);
  p += round16(int64_t(kLayoutMaxTiles) * count_row_width(E, R) * 4);
  ws.tile_err = reinterpret_cast<int32_t*>(p);
  return ws;
}

// An id outside [-1, E) is reported and treated as unused (-1) from here on,
// so that no later kernel can index out of range.
__device__ __forceinline__ int read_expert(const int64_t* __restrict__ p,
                                           int E, int& err) {
  const int64_t v = *p;
  if (v < -1 || v >= E) {
    err |= ERRBIT_EXPERT_RANGE;
    return -1;
  }
  return static_cast<int>(v);
}


// 4 bits of m -> 4 bytes of 0/1 (bit i -> byte i).
__device__ __forceinline__ uint32_t spread4(uint64_t m) {
  return (static_cast<uint32_t>(m & 0xFu) * 0x204081u) & 0x01010101u;
}

// Writes one row of is_token_in_rank (R bytes, byte r = bit r of mask) with
// the widest stores the row's alignment allows (rows start at t * R).
__device__ __forceinline__ void write_rank_row(uint8_t* row, int R, uint64_t mask) {
  if ((R & 15) == 0) {
    for (int i = 0; i < R; i += 16)
      *reinterpret_cast<uint4*>(row + i) =
          make_uint4(spread4(mask >> i), spread4(mask >> (i + 4)),
                     spread4(mask >> (i + 8)), spread4(mask >> (i + 12)));
  } else if ((R & 7) == 0) {
    for (int i = 0; i < R; i += 8)
      *reinterpret_cast<uint2*>(row + i) =
          make_uint2(spread4(mask >> i), spread4(mask >> (i + 4)));
  } else if ((R & 3) == 0) {
    for (int i = 0; i < R; i += 4) *reinterpret_cast<uint32_t*>(row + i) = spread4(mask >> i);
  } else {
    for (int r = 0; r < R; ++r) row[r] = static_cast<uint8_t>((mask >> r) & 1u);
  }
}

// Pairs per unrolled round of a warp: U steps, loads issued before use.
constexpr int kSurveyUnroll = 4;

// One warp step over the selections of whole tokens: lanes [0, TPS*K) hold
// the pairs [base, base + TPS*K) of the tile (lanes past `pe` or past the
// step hold e = -1), so a token's K selections sit in adjacent lanes.  Each
// lane adds its pair to `hist` and reads its token's selections by
// shuffles: the same expert at an earlier k is a repeat; no earlier
// selection on the same rank makes it the token's first on that rank, which
// adds one to s_rank; the token's first lane writes the token's
// destination-rank row.  All lanes call.
__device__ __forceinline__ void survey_step(int e, int lane, int base, int pe, int K,
                                            int TPS, int Eg, int R, int32_t* hist,
                                            uint8_t* itr_tile, int32_t* s_rank,
                                            int& errbits) {
  const int tl = lane / K, kk = lane - tl * K, g0 = tl * K;
  const bool token_live = lane < TPS * K && base + g0 < pe;
  if (e >= 0) atomicAdd(&hist[e], 1);
  const int r = e >= 0 ? e / Eg : -1;
  bool first = true;
  uint64_t mask = 0;
  for (int j = 0; j < K; ++j) {
    // lanes past the step read wrapped lanes; their results are unused
    const int ej = __shfl_sync(0xffffffffu, e, (g0 + j) & 31);
    const int rj = __shfl_sync(0xffffffffu, r, (g0 + j) & 31);
    if (ej < 0) continue;
    if (R <= 64) mask |= uint64_t(1) << rj;
    if (j < kk) {
      if (ej == e) errbits |= ERRBIT_DUP_EXPERT;
      if (rj == r) first = false;
    }
  }
  const bool lead = token_live && kk == 0;
  uint8_t* row = itr_tile + int64_t(base / K + tl) * R;
  if (R <= 64) {
    if (lead) write_rank_row(row, R, mask);
  } else {
    if (lead)
      for (int q = 0; q < R; ++q) row[q] = 0;
    __syncwarp();
    if (e >= 0 && first) row[r] = 1;
  }
  if (e >= 0 && first) atomicAdd(&s_rank[r], 1);
  __syncwarp();
}

// A warp's whole survey of its token-aligned span [tb, te) of a tile.
__device__ __forceinline__ void survey_span(const int64_t* __restrict__ src, int tb, int te,
                                            int K, int E, int R, int lane, int32_t* hist,
                                            uint8_t* itr_tile, int32_t* s_rank, int& errbits) {
  const int TPS = 32 / K, SP = TPS * K, Eg = E / R;
  const int pb = tb * K, pe = te * K;
  for (int b0 = pb; b0 < pe; b0 += SP * kSurveyUnroll) {
    int ev[kSurveyUnroll];
#pragma unroll
    for (int u = 0; u < kSurveyUnroll; ++u) {
      const int p = b0 + u * SP + lane;
      ev[u] = (lane < SP && p < pe) ? read_expert(src + p, E, errbits) : -1;
    }
#pragma unroll
    for (int u = 0; u < kSurveyUnroll; ++u) {
      const int base = b0 + u * SP;
      if (base >= pe) break;
      survey_step(ev[u], lane, base, pe, K, TPS, Eg, R, hist, itr_tile, s_rank, errbits);
    }
  }
}

// ---------------------------------------------------------------------------
// 1. count
// ---------------------------------------------------------------------------
template <bool k16>
__global__ void __launch_bounds__(kLayoutThreads)
    layout_count_kernel(const int64_t* __restrict__ topk_idx, int T, int K,
                        int E, int R, int tile_tokens,
                        int32_t* __restrict__ tile_counts,
                        int32_t* __restrict__ tile_err,
                        uint8_t* __restrict__ is_token_in_rank,
                        int32_t* __restrict__ err) {
  extern __shared__ int32_t smem_i32[];
  __shared__ int32_t s_err;
  const int Wc = count_row_width(E, R);
  int32_t* hist = smem_i32;                  // [Wc]: experts, then ranks
  int32_t* rcnt = hist + padded_experts(E);  // [Rpad]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) s_err = 0;
  for (int e = tid; e < Wc; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  pdl_wait();

  const int tile = blockIdx.x;
  // The call's error word starts at zero here; the assign kernel (which
  // waits for this grid) only ORs bits into it, so a timeout one of its
  // CTAs records is never overwritten.
  if (tile == 0 && tid == 0) *err = 0;
  const int t0 = tile * tile_tokens;
  const int nt = min(tile_tokens, T - t0);
  const int64_t* src = topk_idx + int64_t(t0) * K;
  int bits = 0;
  // Warps take token-aligned spans: expert histogram (shared adds),
  // duplicate experts, destination ranks.
  const int span = (nt + kLayoutWarps - 1) / kLayoutWarps;
  const int tb = min(nt, warp * span), te = min(nt, tb + span);
  survey_span(src, tb, te, K, E, R, lane, hist, is_token_in_rank + int64_t(t0) * R, rcnt,
              bits);
  if (bits) atomicOr(&s_err, bits);
  __syncthreads();

  if (k16) {
    // two 16-bit counts a word, the row padded with zeros to 8 entries
    const int Wr = count_row_entries(E, R, true);
    uint32_t* row = reinterpret_cast<uint32_t*>(tile_counts) + int64_t(tile) * (Wr / 2);
    for (int i = tid; i < Wr / 2; i += blockDim.x) {
      const uint32_t lo = 2 * i < Wc ? uint32_t(hist[2 * i]) : 0u;
      const uint32_t hi = 2 * i + 1 < Wc ? uint32_t(hist[2 * i + 1]) : 0u;
      row[i] = lo | (hi << 16);
    }
  } else {
    for (int e = tid; e < Wc; e += blockDim.x)
      tile_counts[int64_t(tile) * Wc + e] = hist[e];
  }
  if (tid == 0) tile_err[tile] = s_err;
}

// ---------------------------------------------------------------------------
// 2. assign
// ---------------------------------------------------------------------------

// Block-wide exclusive scan of one int per thread (all threads must call).
// s_warp[0..31] may be written again only after a __syncthreads() that
// follows the call (every caller has one before its next use).
__device__ __forceinline__ int block_exclusive_scan(int v, int32_t* s_warp,
                                                    int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
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
  *total = s_warp[nw - 1];
  return warp_excl + x - v;
}

struct AssignSmem {
  // byte offsets into dynamic shared memory
  int bar, ring, whist, start, base, total, rstart, rbase, rtotal, scratch, part, bytes;
  int chunk_rows;
  int row_groups;   // row groups of the column sums (see sum_columns)
};

// Shared-memory plan of the assign kernel; identical on host and device.
// k16: the tile-count rows hold 16-bit counts (count_row_entries).
__host__ __device__ inline AssignSmem assign_smem(int E, int R, int num_tiles, bool k16) {
  const int Epad = padded_experts(E), Rpad = padded_ranks(R);
  const int Wr = count_row_entries(E, R, k16);       // entries a stored row
  const int row_bytes = count_row_bytes(E, R, k16);
  AssignSmem s;
  // column sums: one 16-byte vector of a row a thread (4 or 8 columns); the
  // threads left over take row groups (at most as many as keep the partial
  // sums, int32 per column, within 16 KB)
  const int col_groups = Wr / (k16 ? 8 : 4);
  s.row_groups = col_groups < kAssignThreads ? kAssignThreads / col_groups : 1;
  const int max_groups = 16384 / (8 * Wr);
  if (s.row_groups > max_groups) s.row_groups = max_groups > 1 ? max_groups : 1;
  const int part_bytes = 2 * s.row_groups * Wr * 4;
  // bytes of everything but the count rows (barriers, histograms, scans,
  // partial sums)
  const int other = 16 + kLayoutWarps * E * 4 + ((E + 1 + 3) & ~3) * 4 + 2 * Epad * 4 +
                    ((R + 1 + 3) & ~3) * 4 + 2 * Rpad * 4 + 36 * 4 + part_bytes;
  int rows, nbuf;
  if (num_tiles >= 1 && other + num_tiles * row_bytes <= kAssignSmemBudget) {
    rows = num_tiles;  // the whole matrix in one bulk copy
    nbuf = 1;
  } else {
    rows = kScanChunkBytes / row_bytes;
    if (rows < 1) rows = 1;
    if (num_tiles >= 1 && rows > num_tiles) rows = num_tiles;
    nbuf = 2;
  }
  s.chunk_rows = rows;
  s.bar = 0;                                   // 2 x 8 bytes, padded
  s.ring = 16;                                 // nbuf x rows x row_bytes
  s.whist = s.ring + nbuf * rows * row_bytes;  // kLayoutWarps x E
  s.start = s.whist + kLayoutWarps * E * 4;    // E + 1
  s.base = s.start + ((E + 1 + 3) & ~3) * 4;   // E
  s.total = s.base + Epad * 4;                 // E
  s.rstart = s.total + Epad * 4;               // R + 1
  s.rbase = s.rstart + ((R + 1 + 3) & ~3) * 4; // R
  s.rtotal = s.rbase + Rpad * 4;               // R
  s.scratch = s.rtotal + Rpad * 4;             // 32 + 4
  s.part = s.scratch + 36 * 4;                 // 2 x row_groups x Wr int32
  s.bytes = s.part + part_bytes;
  return s;
}

template <bool k16>
__global__ void __launch_bounds__(kAssignThreads)
    layout_assign_kernel(const int64_t* __restrict__ topk_idx, int T, int K,
                         int E, int R, int A, int tile_tokens, int num_tiles,
                         const int32_t* __restrict__ tile_counts,
                         const int32_t* __restrict__ tile_err,
                         const uint8_t* __restrict__ is_token_in_rank,
                         int32_t* __restrict__ expert_count,
                         int32_t* __restrict__ expert_start,
                         int32_t* __restrict__ expert_end,
                         int32_t* __restrict__ rank_start,
                         int32_t* __restrict__ tokens_per_rank,
                         int32_t* __restrict__ slot_of,
                         int32_t* __restrict__ src_info,
                         int32_t* __restrict__ rank_row_start,
                         int32_t* __restrict__ rank_slot_of,
                         int32_t* __restrict__ rank_src,
                         int32_t* __restrict__ err, int stall_tile,
                         uint64_t wait_ns) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int Epad = padded_experts(E);
  const int Wr = count_row_entries(E, R, k16);
  const int row_bytes = count_row_bytes(E, R, k16);
  const AssignSmem L = assign_smem(E, R, num_tiles, k16);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint8_t* ring = smem + L.ring;
  int32_t* whist = reinterpret_cast<int32_t*>(smem + L.whist);
  int32_t* s_start = reinterpret_cast<int32_t*>(smem + L.start);
  int32_t* s_base = reinterpret_cast<int32_t*>(smem + L.base);
  int32_t* s_total = reinterpret_cast<int32_t*>(smem + L.total);
  int32_t* s_rstart = reinterpret_cast<int32_t*>(smem + L.rstart);
  int32_t* s_rbase = reinterpret_cast<int32_t*>(smem + L.rbase);
  int32_t* s_rtotal = reinterpret_cast<int32_t*>(smem + L.rtotal);
  int32_t* s_scr = reinterpret_cast<int32_t*>(smem + L.scratch);
  int32_t* s_part = reinterpret_cast<int32_t*>(smem + L.part);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int tile = blockIdx.x;
  const bool has_tile = tile < num_tiles;
  int2* src_info2 = reinterpret_cast<int2*>(src_info);

  for (int i = tid; i < kLayoutWarps * E; i += blockDim.x) whist[i] = 0;
  for (int e = tid; e < E; e += blockDim.x) {
    s_base[e] = 0;
    s_total[e] = 0;
  }
  for (int r = tid; r < R; r += blockDim.x) {
    s_rbase[r] = 0;
    s_rtotal[r] = 0;
  }
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();

  // Stream the tile-count matrix through two shared-memory buffers.  The
  // CTA numbered stall_tile (a self-test; -1 otherwise) issues no copy, so
  // its first wait runs out.
  const int rows = L.chunk_rows;
  const int nchunks = num_tiles > 0 ? (num_tiles + rows - 1) / rows : 0;
  const bool stall = tile == stall_tile;
  int issued = 0;   // chunks whose copy thread 0 has issued
  auto issue = [&](int ch) {
    if (stall) return;
    const int r0 = ch * rows;
    const int n = min(rows, num_tiles - r0);
    const uint32_t bytes = uint32_t(n) * uint32_t(row_bytes);
    mbar_arrive_expect_tx(&bar[ch & 1], bytes);
    bulk_load(ring + (ch & 1) * rows * row_bytes,
              reinterpret_cast<const uint8_t*>(tile_counts) + int64_t(r0) * row_bytes, bytes,
              &bar[ch & 1]);
    issued = ch + 1;
  };
  if (tid == 0) {
    if (nchunks > 0) issue(0);
    if (nchunks > 1) issue(1);
  }

  // Pass 1 (overlaps the copies): per-warp histogram of this tile.  Warp w
  // < kLayoutWarps owns the contiguous pairs [pb, pe); the other warps own
  // none (they join the column sums, scans and stores below).
  int t0 = 0, P = 0, pb = 0, pe = 0;
  int ignored = 0;
  if (has_tile) {
    t0 = tile * tile_tokens;
    P = min(tile_tokens, T - t0) * K;
    const int span = (P + kLayoutWarps - 1) / kLayoutWarps;
    pb = min(P, warp * span);
    pe = min(P, pb + span);
  }
  const int64_t* src = topk_idx + int64_t(t0) * K;
  int32_t* my = whist + warp * E;
  for (int b0 = pb; b0 < pe; b0 += 32 * kSurveyUnroll) {
    int ev[kSurveyUnroll];
#pragma unroll
    for (int u = 0; u < kSurveyUnroll; ++u) {
      const int p = b0 + u * 32 + lane;
      ev[u] = p < pe ? read_expert(src + p, E, ignored) : -1;
    }
#pragma unroll
    for (int u = 0; u < kSurveyUnroll; ++u)
      if (ev[u] >= 0) atomicAdd(&my[ev[u]], 1);
  }

  // Per expert: rows of earlier tiles (this tile's base) and of all tiles.
  int failed = -1;
  for (int ch = 0; ch < nchunks; ++ch) {
    if (tid == 0) s_scr[32] = mbar_wait(&bar[ch & 1], (ch >> 1) & 1, wait_ns);
    __syncthreads();
    if (!s_scr[32]) {
      failed = ch;
      break;
    }
    const int r0 = ch * rows;
    const int n = min(rows, num_tiles - r0);
    const uint8_t* buf = ring + (ch & 1) * rows * row_bytes;
    // Column sums -- all rows (totals) and rows of earlier tiles (this
    // tile's base) -- one 16-byte vector of each row a thread (4 32-bit or
    // 8 16-bit counts), rows split into L.row_groups groups so that many
    // loads are in flight; the groups' partial sums then meet in shared
    // memory.
    {
      const int nb = min(n, max(0, tile - r0));   // rows of earlier tiles
      constexpr int kCols = k16 ? 8 : 4;          // columns a vector
      const int col_groups = Wr / kCols, G = L.row_groups;
      const int per = (n + G - 1) / G;
      for (int w = tid; w < col_groups * G; w += blockDim.x) {
        const int cgi = w % col_groups, g = w / col_groups;
        const int ra = g * per, rb = min(n, ra + per);
        int tot[kCols], bas[kCols];
#pragma unroll
        for (int j = 0; j < kCols; ++j) tot[j] = bas[j] = 0;
#pragma unroll 4
        for (int r = ra; r < rb; ++r) {
          const uint4 v = *reinterpret_cast<const uint4*>(buf + r * row_bytes + cgi * 16);
          int c[kCols];
          if constexpr (k16) {
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              c[2 * q] = int(wv[q] & 0xFFFFu);
              c[2 * q + 1] = int(wv[q] >> 16);
            }
          } else {
            c[0] = int(v.x);
            c[1] = int(v.y);
            c[2] = int(v.z);
            c[3] = int(v.w);
          }
#pragma unroll
          for (int j = 0; j < kCols; ++j) tot[j] += c[j];
          if (r < nb) {
#pragma unroll
            for (int j = 0; j < kCols; ++j) bas[j] += c[j];
          }
        }
#pragma unroll
        for (int j = 0; j < kCols; j += 4) {
          *reinterpret_cast<int4*>(s_part + (g * Wr + cgi * kCols + j)) =
              make_int4(tot[j], tot[j + 1], tot[j + 2], tot[j + 3]);
          *reinterpret_cast<int4*>(s_part + ((G + g) * Wr + cgi * kCols + j)) =
              make_int4(bas[j], bas[j + 1], bas[j + 2], bas[j + 3]);
        }
      }
      __syncthreads();
      for (int c = tid; c < Wr; c += blockDim.x) {
        const bool is_e = c < E, is_r = c >= Epad && c - Epad < R;
        if (!is_e && !is_r) continue;
        int tot = 0, bas = 0;
        for (int g = 0; g < G; ++g) {
          tot += s_part[g * Wr + c];
          bas += s_part[(G + g) * Wr + c];
        }
        if (is_e) {
          s_base[c] += bas;
          s_total[c] += tot;
        } else {
          s_rbase[c - Epad] += bas;
          s_rtotal[c - Epad] += tot;
        }
      }
    }
    __syncthreads();
    if (tid == 0 && ch + 2 < nchunks) issue(ch + 2);
  }
  if (failed >= 0) {
    // A copy did not land in time: report, wait (bounded) for the copies
    // this CTA issued that are still in flight -- chunks [failed, issued) --
    // and leave without writing rows.  Should one of those waits give up
    // too, the copy may still land in this SM's shared memory after the CTA
    // ends; that is reported as a bit of its own.
    if (tid == 0) {
      record_error(err, ERRBIT_TIMEOUT);
      for (int ch = failed; ch < issued; ++ch)
        if (!mbar_wait(&bar[ch & 1], (ch >> 1) & 1, kWaitTimeoutNs))
          record_error(err, ERRBIT_TIMEOUT_PENDING);
    }
    return;
  }

  // Aligned exclusive scan over experts: each segment rounded up to a
  // multiple of A; the valid rows of expert e end at start + count.
  const int per = (E + blockDim.x - 1) / blockDim.x;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int local = 0;
  for (int e = e0; e < e1; ++e) local += (s_total[e] + A - 1) / A * A;
  int used = 0;
  int run = block_exclusive_scan(local, s_scr, &used);
  for (int e = e0; e < e1; ++e) {
    s_start[e] = run;
    run += (s_total[e] + A - 1) / A * A;
  }
  if (tid == 0) s_start[E] = used;
  __syncthreads();

  if (has_tile) {
    // Per-warp bases: aligned expert start + rows of earlier tiles + rows of
    // earlier warps of this tile.
    for (int e = tid; e < E; e += blockDim.x) {
      int r = s_start[e] + s_base[e];
      for (int w = 0; w < kLayoutWarps; ++w) {
        const int c = whist[w * E + e];
        whist[w * E + e] = r;
        r += c;
      }
    }
    __syncthreads();

    // Pass 2: rows, in (t, k) order within each expert.
    const uint32_t lt = lanemask_lt();
    for (int b0 = pb; b0 < pe; b0 += 32 * kSurveyUnroll) {
      int ev[kSurveyUnroll];
#pragma unroll
      for (int u = 0; u < kSurveyUnroll; ++u) {
        const int p = b0 + u * 32 + lane;
        ev[u] = p < pe ? read_expert(src + p, E, ignored) : -1;
      }
#pragma unroll
      for (int u = 0; u < kSurveyUnroll; ++u) {
        if (b0 + u * 32 >= pe) break;
        const int p = b0 + u * 32 + lane;
        const int e = ev[u];
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        int slot = -1;
        if (e >= 0) slot = my[e] + __popc(peers & lt);
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
        __syncwarp();
        if (p < pe) {
          slot_of[int64_t(t0) * K + p] = slot;
          if (slot >= 0) {
            const int tl = p / K;
            src_info2[slot] = make_int2(t0 + tl, p - tl * K);
          }
        }
      }
    }
  }

  // Published per-expert arrays (CTA 0) and the error word.
  if (tile == 0) {
    for (int e = tid; e < E; e += blockDim.x) {
      expert_count[e] = s_total[e];
      expert_start[e] = s_start[e];
      expert_end[e] = s_start[e] + s_total[e];
    }
    if (tid == 0) expert_start[E] = s_start[E];
    const int Eg = E / R;
    for (int r = tid; r <= R; r += blockDim.x) rank_start[r] = s_start[r * Eg];
    int bits = 0;
    for (int c = tid; c < num_tiles; c += blockDim.x) bits |= tile_err[c];
    if (tid == 0) s_scr[33] = 0;
    __syncthreads();
    if (bits) atomicOr(&s_scr[33], bits);
    __syncthreads();
    // OR-ed in: the count kernel cleared the word, and another CTA may
    // already have recorded a timeout.  With no tokens there was no count
    // kernel and this is the grid's only CTA, so it stores.
    if (tid == 0) {
      if (num_tiles > 0) {
        if (s_scr[33]) atomicOr(err, s_scr[33]);
      } else {
        *err = s_scr[33];
      }
    }
  }

  // Tokens per destination rank (totals of the rank columns).
  if (tile == 0)
    for (int r = tid; r < R; r += blockDim.x) tokens_per_rank[r] = s_rtotal[r];

  // Optional rank rows: rank r owns rows [rank_row_start[r],
  // rank_row_start[r+1]), one per token sent to it, in token order.
  if (rank_slot_of != nullptr) {
    const int rper = (R + blockDim.x - 1) / blockDim.x;
    const int q0 = min(R, tid * rper), q1 = min(R, q0 + rper);
    int rl = 0;
    for (int q = q0; q < q1; ++q) rl += s_rtotal[q];
    int rows_all = 0;
    int rrun = block_exclusive_scan(rl, s_scr, &rows_all);
    for (int q = q0; q < q1; ++q) {
      s_rstart[q] = rrun;
      rrun += s_rtotal[q];
    }
    if (tid == 0) s_rstart[R] = rows_all;
    __syncthreads();
    if (tile == 0)
      for (int q = tid; q <= R; q += blockDim.x) rank_row_start[q] = s_rstart[q];
    if (has_tile) {
      // one warp per rank: ballot over the tile's tokens, 32 at a time
      const int nt = min(tile_tokens, T - t0);
      const uint32_t lt = lanemask_lt();
      for (int q = warp; q < R; q += nwarps) {
        int run = s_rstart[q] + s_rbase[q];
        for (int c0 = 0; c0 < nt; c0 += 32) {
          const int t = t0 + c0 + lane;
          const bool in_tile = c0 + lane < nt;
          const bool flag = in_tile && is_token_in_rank[int64_t(t) * R + q] != 0;
          const uint32_t m = __ballot_sync(0xffffffffu, flag);
          const int row = run + __popc(m & lt);
          if (in_tile) rank_slot_of[int64_t(t) * R + q] = flag ? row : -1;
          if (flag) rank_src[row] = t;
          run += __popc(m);
        }
      }
    }
  }

  // Alignment padding rows carry no token (one warp per expert at a time).
  for (int e = blockIdx.x * nwarps + warp; e < E; e += gridDim.x * nwarps) {
    const int s0 = s_start[e] + s_total[e], s1 = s_start[e + 1];
    for (int s = s0 + lane; s < s1; s += 32) src_info2[s] = make_int2(-1, -1);
  }
}


// ---------------------------------------------------------------------------
// small inputs: one launch
// ---------------------------------------------------------------------------
// When T * K is small (decode batches), the two-launch path is all latency.
// Here every CTA surveys the whole input itself, one token per thread --
// counts of the tokens before its own range, within it and after it -- so
// that no CTA waits for another; then the same aligned scan as the assign
// kernel, rows for its own few tokens in (t, k) order, rank rows and
// padding.  The rows are the same as the two-launch path's.
struct SmallSmem {
  int idx, hist, start, total, base, rcnt, rstart, scr, own, rows, bytes;
};

// Shared-memory plan of the one-launch layout for `pairs` (t, k) pairs
// (the route array is sized to the call, not to the largest input this
// path takes: at decode that halves the kernel's shared memory, and the
// step measured 0.4-0.9 us faster); with row_bytes > 0 it ends with room
// for the rows of the CTA's own tokens (fused dispatch, staged).
// Every region is a multiple of 16 bytes, so the staged rows start on a
// 16-byte boundary.
__host__ __device__ inline SmallSmem small_smem(int E, int R, int pairs, int64_t row_bytes = 0) {
  const int Epad = padded_experts(E), Rpad = padded_ranks(R);
  SmallSmem s;
  int o = 0;
  s.idx = o;    o += (pairs * 4 + 15) & ~15;       // the routes, checked, packed
  s.hist = o;   o += 3 * Epad * 4;                 // counts: earlier, own, later tokens
  s.start = o;  o += ((E + 1 + 3) & ~3) * 4;
  s.total = o;  o += Epad * 4;
  s.base = o;   o += Epad * 4;                     // next row of each expert
  s.rcnt = o;   o += 3 * Rpad * 4;                 // rank counts, same regions
  s.rstart = o; o += ((R + 1 + 3) & ~3) * 4;
  s.scr = o;    o += 36 * 4;                       // scan scratch, [33] = errors
  s.own = o;    o += kSmallOwnPairs * 4;           // rows of this CTA's pairs
  s.rows = o;   o += static_cast<int>(row_bytes);  // staged x rows (16-byte aligned)
  s.bytes = o;
  return s;
}

// n / d for 0 <= n < 2^16 and 1 <= d <= 2048 by a multiply-high with
// magic = ceil(2^32 / d) (magic 0 stands for d = 1): the product's error,
// below n / 2^32 < 2^-16, never reaches the next multiple of 1/d.
__host__ __device__ inline uint32_t div_magic(uint32_t d) {
  return d == 1 ? 0u : uint32_t(0xFFFFFFFFu / d + 1u);
}
__device__ __forceinline__ int small_div(int n, uint32_t magic) {
  return magic == 0 ? n : int(__umulhi(uint32_t(n), magic));
}

// A selection packed for the survey: expert in the low 16 bits, its
// destination rank in the high 16 (both below 2048), -1 if unused.
__device__ __forceinline__ int32_t pack_route(int e, uint32_t eg_magic) {
  return e < 0 ? -1 : (e | (small_div(e, eg_magic) << 16));
}
__device__ __forceinline__ int route_expert(int32_t v) { return v < 0 ? -1 : (v & 0xFFFF); }

// CTAs of the one-launch layout (each owns about T / kSmallLayoutCtas tokens).
constexpr int kSmallLayoutCtas = kLayoutMaxTiles;

// kMode: 0 layout only; 1 and 2 also dispatch each CTA's own tokens, as
// bf16 rows (1) or E4M3 rows with row-major 1x128 scales (2) -- the same
// rows and values as dispatch_bf16_kernel / dispatch_fp8_kernel write.
template <int kMode>
__global__ void __launch_bounds__(kSmallThreads)
    layout_small_kernel(const int64_t* __restrict__ topk_idx, int T, int K, int E,
                        int R, int A, SmallDispatch d, int staged,
                        uint8_t* __restrict__ is_token_in_rank,
                        int32_t* __restrict__ expert_count,
                        int32_t* __restrict__ expert_start,
                        int32_t* __restrict__ expert_end,
                        int32_t* __restrict__ rank_start,
                        int32_t* __restrict__ tokens_per_rank,
                        int32_t* __restrict__ slot_of,
                        int32_t* __restrict__ src_info,
                        int32_t* __restrict__ rank_row_start,
                        int32_t* __restrict__ rank_slot_of,
                        int32_t* __restrict__ rank_src,
                        int32_t* __restrict__ err) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int Epad = padded_experts(E), Rpad = padded_ranks(R);
  const int64_t row_bytes = int64_t(d.H) * (kMode != 0 ? 2 : 0);
  const int tt = (T + gridDim.x - 1) / gridDim.x;
  const SmallSmem L = small_smem(E, R, T * K, staged ? tt * row_bytes : 0);
  int32_t* s_idx = reinterpret_cast<int32_t*>(smem + L.idx);      // [T * K]
  int32_t* hist = reinterpret_cast<int32_t*>(smem + L.hist);      // [3][Epad]
  int32_t* s_start = reinterpret_cast<int32_t*>(smem + L.start);
  int32_t* s_total = reinterpret_cast<int32_t*>(smem + L.total);
  int32_t* s_base = reinterpret_cast<int32_t*>(smem + L.base);
  int32_t* rcnt = reinterpret_cast<int32_t*>(smem + L.rcnt);      // [3][Rpad]
  int32_t* s_rstart = reinterpret_cast<int32_t*>(smem + L.rstart);
  int32_t* s_scr = reinterpret_cast<int32_t*>(smem + L.scr);
  int32_t* s_own = reinterpret_cast<int32_t*>(smem + L.own);       // [kSmallOwnPairs]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int2* src_info2 = reinterpret_cast<int2*>(src_info);

  for (int i = tid; i < 3 * Epad; i += blockDim.x) hist[i] = 0;
  for (int i = tid; i < 3 * Rpad; i += blockDim.x) rcnt[i] = 0;
  if (tid == 0) s_scr[33] = 0;
  __syncthreads();
  pdl_wait();

  // This CTA's tokens [ctb, cte).
  const int ctb = min(T, int(blockIdx.x) * tt), cte = min(T, ctb + tt);
  const int Eg = E / R;
  const uint32_t eg_magic = div_magic(uint32_t(Eg));

  // Fused dispatch with staged rows: the CTA's own x rows (contiguous) are
  // copied into shared memory now, 16 bytes a thread at a time
  // asynchronously, so that their DRAM latency passes while the layout is
  // computed.  (Per-thread copies rather than one bulk copy: their
  // completion needs no flag to wait on, so this kernel has no wait that
  // could give up.)
  const uint32_t stage_bytes = uint32_t((cte - ctb) * row_bytes);
  if (kMode != 0 && staged && stage_bytes > 0) {
    const uint8_t* src = reinterpret_cast<const uint8_t*>(d.x) + ctb * row_bytes;
    for (uint32_t o = uint32_t(tid) * 16; o < stage_bytes; o += blockDim.x * 16)
      cp_async16(smem + L.rows + o, src + o);
    cp_async_commit();
  }

  // The whole input, range-checked (an id outside [-1, E) is reported and
  // read as -1), in shared memory, each selection packed with its
  // destination rank: one pass of independent loads.  The rank rows of this
  // CTA's tokens are cleared meanwhile (set per rank below).
  int errbits = 0;
#pragma unroll 4
  for (int i = tid; i < T * K; i += blockDim.x)
    s_idx[i] = pack_route(read_expert(topk_idx + i, E, errbits), eg_magic);
  for (int i = tid; i < (cte - ctb) * R; i += blockDim.x)
    is_token_in_rank[int64_t(ctb) * R + i] = 0;
  __syncthreads();

  // Survey, one pair a thread (thread = (token slot, k), so no division per
  // pair): the pair adds to its region's expert count (tokens before,
  // inside and after this CTA's range) and reads its token's earlier
  // selections from shared memory: the same expert again is a repeat; no
  // earlier selection on the same rank makes it the token's first on that
  // rank, which adds one to the region's rank count and, for this CTA's own
  // tokens, sets the rank-row flag.
  const int tps = blockDim.x / K;               // tokens per pass
  const int sv_t = tid / K, sv_k = tid - sv_t * K;
  for (int t = sv_t; sv_t < tps && t < T; t += tps) {
    const int32_t* tok = s_idx + t * K;
    const int32_t v = tok[sv_k];
    if (v < 0) continue;
    bool first = true;
    for (int j = 0; j < sv_k; ++j) {
      const int32_t u = tok[j];
      if (u < 0) continue;
      if (u == v) errbits |= ERRBIT_DUP_EXPERT;
      if ((u >> 16) == (v >> 16)) first = false;
    }
    const int e = v & 0xFFFF, r = v >> 16;
    const int region = t < ctb ? 0 : (t < cte ? 1 : 2);
    atomicAdd(&hist[region * Epad + e], 1);
    if (first) {
      atomicAdd(&rcnt[region * Rpad + r], 1);
      if (region == 1) is_token_in_rank[int64_t(t) * R + r] = 1;
    }
  }
  if (errbits) atomicOr(&s_scr[33], errbits);
  __syncthreads();

  // Per-expert totals and the aligned exclusive scan over experts (each
  // thread sums the three regions of its own experts).
  const int per = (E + blockDim.x - 1) / blockDim.x;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int local = 0;
  for (int e = e0; e < e1; ++e) {
    const int c = hist[e] + hist[Epad + e] + hist[2 * Epad + e];
    s_total[e] = c;
    local += (c + A - 1) / A * A;
  }
  int used = 0;
  int run = block_exclusive_scan(local, s_scr, &used);
  for (int e = e0; e < e1; ++e) {
    s_start[e] = run;
    s_base[e] = run + hist[e];    // after the rows of earlier tokens
    run += (s_total[e] + A - 1) / A * A;
  }
  if (tid == 0) s_start[E] = used;
  __syncthreads();

  // Rows of this CTA's tokens (warp 0, 32 pairs a step, in (t, k) order).
  if (warp == 0) {
    const int32_t* src = s_idx + ctb * K;
    const int pe = (cte - ctb) * K;
    const uint32_t lt = lanemask_lt();
    for (int b0 = 0; b0 < pe; b0 += 32) {
      const int p = b0 + lane;
      const int e = p < pe ? route_expert(src[p]) : -1;
      const uint32_t peers = __match_any_sync(0xffffffffu, e);
      int slot = -1;
      if (e >= 0) slot = s_base[e] + __popc(peers & lt);
      __syncwarp();
      if (e >= 0 && lane == __ffs(peers) - 1) s_base[e] += __popc(peers);
      __syncwarp();
      if (p < pe) {
        slot_of[int64_t(ctb) * K + p] = slot;
        if (slot >= 0) {
          const int tl = p / K;
          src_info2[slot] = make_int2(ctb + tl, p - tl * K);
        }
        if (kMode != 0) {
          s_own[p] = slot;
          if (slot >= 0 && d.w != nullptr && d.recv_w != nullptr)
            d.recv_w[slot] = d.w[int64_t(ctb) * K + p];
        }
      }
    }
  }

  // Published per-expert and per-rank arrays (CTA 0, which saw every pair).
  if (blockIdx.x == 0) {
    for (int e = tid; e < E; e += blockDim.x) {
      expert_count[e] = s_total[e];
      expert_start[e] = s_start[e];
      expert_end[e] = s_start[e] + s_total[e];
    }
    if (tid == 0) {
      expert_start[E] = s_start[E];
      // this launch has no waits and no other writer of the word: the store
      // both clears it and publishes the call's routing errors
      *err = s_scr[33];
    }
    for (int r = tid; r <= R; r += blockDim.x) rank_start[r] = s_start[r * Eg];
    for (int r = tid; r < R; r += blockDim.x)
      tokens_per_rank[r] = rcnt[r] + rcnt[Rpad + r] + rcnt[2 * Rpad + r];
  }

  // Optional rank rows, in token order within each rank.
  if (rank_slot_of != nullptr) {
    const int rper = (R + blockDim.x - 1) / blockDim.x;
    const int q0 = min(R, tid * rper), q1 = min(R, q0 + rper);
    int rl = 0;
    for (int q = q0; q < q1; ++q) rl += rcnt[q] + rcnt[Rpad + q] + rcnt[2 * Rpad + q];
    int rows_all = 0;
    int rrun = block_exclusive_scan(rl, s_scr, &rows_all);
    for (int q = q0; q < q1; ++q) {
      s_rstart[q] = rrun;
      rrun += rcnt[q] + rcnt[Rpad + q] + rcnt[2 * Rpad + q];
    }
    if (tid == 0) s_rstart[R] = rows_all;
    __syncthreads();  // also orders this CTA's rank-row bytes before the reads
    if (blockIdx.x == 0)
      for (int q = tid; q <= R; q += blockDim.x) rank_row_start[q] = s_rstart[q];
    const int nt = cte - ctb;
    const uint32_t lt = lanemask_lt();
    for (int q = warp; q < R; q += kSmallWarps) {
      int rr = s_rstart[q] + rcnt[q];
      for (int c0 = 0; c0 < nt; c0 += 32) {
        const int t = ctb + c0 + lane;
        const bool in_range = c0 + lane < nt;
        const bool flag = in_range && is_token_in_rank[int64_t(t) * R + q] != 0;
        const uint32_t m = __ballot_sync(0xffffffffu, flag);
        const int row = rr + __popc(m & lt);
        if (in_range) rank_slot_of[int64_t(t) * R + q] = flag ? row : -1;
        if (flag) rank_src[row] = t;
        rr += __popc(m);
      }
    }
  }

  // Alignment padding rows carry no token (one warp per expert at a time).
  for (int e = blockIdx.x * kSmallWarps + warp; e < E; e += gridDim.x * kSmallWarps) {
    const int s0 = s_start[e] + s_total[e], s1 = s_start[e + 1];
    for (int s = s0 + lane; s < s1; s += 32) src_info2[s] = make_int2(-1, -1);
  }

  if (kMode == 0) return;
  // Dispatch of this CTA's own tokens to the rows just assigned, from the
  // staged rows in shared memory (or from x when they did not fit).
  if (staged && stage_bytes > 0) cp_async_wait_all();
  __syncthreads();
  const int nt = cte - ctb;
  const int nvec = d.H >> 3;
  const uint4* srows = reinterpret_cast<const uint4*>(smem + L.rows);  // staged rows
  if (kMode == 1) {
    uint4* rx = static_cast<uint4*>(d.recv_x);
    for (int i = 0; i < nt; ++i) {
      const uint4* row = d.x + int64_t(ctb + i) * nvec;
      const uint4* srow = srows + int64_t(i) * nvec;
      for (int v = tid; v < nvec; v += blockDim.x) {
        const uint4 r = staged ? srow[v] : ld_stream_u4(row + v);
        for (int k = 0; k < K; ++k) {
          const int sl = s_own[i * K + k];
          if (sl >= 0) rx[int64_t(sl) * nvec + v] = r;
        }
      }
    }
  } else {
    // 8 aligned lanes per 128-channel block (blockDim is a multiple of 32)
    uint8_t* rq = static_cast<uint8_t*>(d.recv_x);
    const int n16 = d.H >> 4, nblk = d.H >> 7;
    for (int i = 0; i < nt; ++i) {
      const uint4* row = d.x + int64_t(ctb + i) * nvec;
      const uint4* srow = srows + int64_t(i) * nvec;
      for (int base = 0; base < n16; base += blockDim.x) {
        const int u = base + tid;
        const bool active = u < n16;
        uint4 r0 = make_uint4(0, 0, 0, 0), r1 = r0;
        if (active) {
          if (staged) {
            r0 = srow[2 * u];
            r1 = srow[2 * u + 1];
          } else {
            r0 = ld_stream_u4(row + 2 * u);
            r1 = ld_stream_u4(row + 2 * u + 1);
          }
        }
        uint4 q;
        float scale;
        quantize_group16(r0, r1, &q, &scale);
        if (!active) continue;
        const bool leader = (tid & 7) == 0;
        for (int k = 0; k < K; ++k) {
          const int sl = s_own[i * K + k];
          if (sl < 0) continue;
          *reinterpret_cast<uint4*>(rq + int64_t(sl) * d.H + int64_t(u) * 16) = q;
          if (leader) d.recv_scale[int64_t(sl) * nblk + (u >> 3)] = scale;
        }
      }
    }
  }
}

static int count_smem(int E, int R, int K) {
  (void)K;
  return count_row_width(E, R) * 4;
}

cudaError_t prepare_layout_kernels() {
  const int optin = device_info().max_smem_optin;
  cudaError_t st = allow_max_dynamic_smem(layout_count_kernel<false>, optin);
  if (st == cudaSuccess) st = allow_max_dynamic_smem(layout_count_kernel<true>, optin);
  if (st == cudaSuccess) st = allow_max_dynamic_smem(layout_small_kernel<0>, optin);
  if (st == cudaSuccess) st = allow_max_dynamic_smem(layout_small_kernel<1>, optin);
  if (st == cudaSuccess) st = allow_max_dynamic_smem(layout_small_kernel<2>, optin);
  if (st == cudaSuccess) st = allow_max_dynamic_smem(layout_assign_kernel<false>, optin);
  if (st != cudaSuccess) return st;
  return allow_max_dynamic_smem(layout_assign_kernel<true>, optin);
}

bool layout_is_small(int64_t T, int K, int E) {
  return T * K <= kSmallLayoutPairs && E <= kSmallLayoutMaxExperts;
}

int assign_grid(int tiles, int E) {
  int grid = tiles > 0 ? tiles : 1;
  const int pad_blocks = E < kLayoutMaxTiles ? E : kLayoutMaxTiles;
  if (tiles > 0 && grid < pad_blocks) grid = pad_blocks;
  return grid;
}

cudaError_t launch_layout(const LayoutArgs& a, cudaStream_t stream) {
  if (layout_is_small(a.T, a.K, a.E)) {
    return launch_pdl(layout_small_kernel<0>, dim3(kSmallLayoutCtas), dim3(kSmallThreads),
                      small_smem(a.E, a.R, a.T * a.K).bytes, stream, a.topk_idx, a.T, a.K,
                      a.E, a.R, a.A, SmallDispatch{}, 0, a.is_token_in_rank, a.expert_count,
                      a.expert_start, a.expert_end, a.rank_start, a.tokens_per_rank,
                      a.slot_of, a.src_info, a.rank_row_start, a.rank_slot_of, a.rank_src,
                      a.err);
  }
  const int tiles = a.T > 0 ? a.geom.num_tiles : 0;
  const int tt = a.geom.tile_tokens;
  // 16-bit tile counts when no count can exceed them (a tile's pairs)
  const bool k16 = int64_t(tt) * a.K <= 0xFFFF;
  cudaError_t st;
  if (tiles > 0) {
    st = launch_pdl(k16 ? layout_count_kernel<true> : layout_count_kernel<false>, dim3(tiles),
                    dim3(kLayoutThreads), count_smem(a.E, a.R, a.K), stream, a.topk_idx, a.T,
                    a.K, a.E, a.R, tt, a.ws.tile_counts, a.ws.tile_err, a.is_token_in_rank,
                    a.err);
    if (st != cudaSuccess) return st;
  }
  // With no tokens there are no tiles: one CTA still publishes the empty
  // layout (zero counts and offsets).
  const AssignSmem sm = assign_smem(a.E, a.R, tiles, k16);
  const int grid = assign_grid(tiles, a.E);
  return launch_pdl(k16 ? layout_assign_kernel<true> : layout_assign_kernel<false>, dim3(grid),
                    dim3(kAssignThreads),
                    sm.bytes, stream, a.topk_idx, a.T, a.K, a.E, a.R, a.A, tt,
                    tiles, a.ws.tile_counts, a.ws.tile_err,
                    static_cast<const uint8_t*>(a.is_token_in_rank), a.expert_count,
                    a.expert_start, a.expert_end, a.rank_start, a.tokens_per_rank,
                    a.slot_of, a.src_info, a.rank_row_start, a.rank_slot_of,
                    a.rank_src, a.err, a.stall_tile, a.wait_ns);
}

// Rows of the pairs one CTA of the one-launch layout owns, at most.
static bool small_fusable(int T, int K) {
  const int tt = (T + kSmallLayoutCtas - 1) / kSmallLayoutCtas;
  return tt * K <= kSmallOwnPairs;
}

cudaError_t launch_layout_dispatch(const LayoutArgs& la, const DispatchArgs& da,
                                   cudaStream_t stream) {
  const bool fuse = la.T > 0 && layout_is_small(la.T, la.K, la.E) && small_fusable(la.T, la.K) &&
                    da.x_q == nullptr && !da.scale_col_major;
  if (!fuse) {
    cudaError_t st = launch_layout(la, stream);
    return st != cudaSuccess ? st : launch_dispatch(da, stream);
  }
  SmallDispatch d;
  d.x = static_cast<const uint4*>(da.x);
  d.w = da.topk_weights;
  d.recv_x = da.recv_x;
  d.recv_scale = da.recv_scale;
  d.recv_w = da.recv_w;
  d.H = da.H;
  auto kern = da.fp8 ? layout_small_kernel<2> : layout_small_kernel<1>;
  // Stage the CTAs' own x rows in shared memory when they fit beside the
  // layout's arrays.
  const int tt = (la.T + kSmallLayoutCtas - 1) / kSmallLayoutCtas;
  const int64_t staged_bytes =
      small_smem(la.E, la.R, la.T * la.K, int64_t(tt) * da.H * 2).bytes;
  const bool staged = staged_bytes <= kSmallStageBudget &&
                      (reinterpret_cast<uintptr_t>(da.x) & 15) == 0;
  const int smem = staged ? int(staged_bytes) : small_smem(la.E, la.R, la.T * la.K).bytes;
  cudaError_t st = launch_pdl(kern, dim3(kSmallLayoutCtas), dim3(kSmallThreads),
                              smem, stream, la.topk_idx, la.T, la.K,
                              la.E, la.R, la.A, d, int(staged), la.is_token_in_rank, la.expert_count,
                              la.expert_start, la.expert_end, la.rank_start,
                              la.tokens_per_rank, la.slot_of, la.src_info, la.rank_row_start,
                              la.rank_slot_of, la.rank_src, la.err);
  if (st != cudaSuccess || !da.zero_padding) return st;
  DispatchArgs z = da;   // the alignment gap rows, as ep_dispatch clears them
  z.T = 0;
  return launch_dispatch(z, stream);
}

}  // namespace ep

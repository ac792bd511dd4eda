// Non-expanded (destination-major) stage ("Deep Dive - DeepEP": "Why expert
// parallelism needs a communication layer" -- a token travels once to each
// selected destination rank and an optional expansion then makes one slot
// per expert; "Dispatch: layout, move, and epilogue" -- in non-expanded
// mode a received row is a source token with its top-k metadata; "GPU
// Microarchitecture: DeepEP from First Principles" 2.1 -- receive buffer ->
// expert buffer, 1.2 -- expert-major -> destination-major -> token-major).
//
// The rank rows come from the layout (rank_slot_of, token order within each
// rank).  All kernels: 16-byte vectors, bf16 rows; a token's row is split
// over one or more CTAs (grid.y), expand also gives each CTA several tokens.
#include "ep_device.cuh"
#include "ep_internal.h"

namespace ep {

// The token's destination ranks in ascending order, compacted by the calling
// warp: s_rank[i], s_row[i] for i < *s_n (a token reaches at most
// min(K, R) <= 32 ranks).  All 32 lanes call.
__device__ __forceinline__ void warp_rank_rows(const int32_t* __restrict__ rank_slot_of,
                                               int t, int R, int32_t* s_rank,
                                               int32_t* s_row, int* s_n) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = lanemask_lt();
  int n = 0;
  for (int c0 = 0; c0 < R; c0 += 32) {
    const int r = c0 + lane;
    const int row = r < R ? rank_slot_of[int64_t(t) * R + r] : -1;
    const uint32_t m = __ballot_sync(0xffffffffu, row >= 0);
    if (row >= 0) {
      const int pos = n + __popc(m & lt);
      if (pos < 32) {
        s_rank[pos] = r;
        s_row[pos] = row;
      }
    }
    n += __popc(m);
  }
  if (lane == 0) *s_n = n < 32 ? n : 32;
}

// As above by warp 0; all threads of the block call and the block is
// synchronised after.
__device__ __forceinline__ void token_rank_rows(const int32_t* __restrict__ rank_slot_of,
                                                int t, int R, int32_t* s_rank,
                                                int32_t* s_row, int* s_n) {
  if (threadIdx.x < 32) warp_rank_rows(rank_slot_of, t, R, s_rank, s_row, s_n);
  __syncthreads();
}

// ---------------------------------------------------------------------------
// dispatch to ranks: rank_x[row(t, r)] = x[t] and the row's top-k metadata
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(512)
    dispatch_ranks_kernel(const uint4* __restrict__ x,
                          const int64_t* __restrict__ topk_idx,
                          const float* __restrict__ w,
                          const int32_t* __restrict__ rank_slot_of, int nvec,
                          int K, int E, int R, uint4* __restrict__ rank_x,
                          int32_t* __restrict__ rank_topk_idx,
                          float* __restrict__ rank_topk_w) {
  __shared__ int32_t s_rank[32], s_row[32];
  __shared__ int s_n;
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  pdl_wait();
  const uint4* row = x + int64_t(t) * nvec;
  const int v0 = first_vec();
  uint4 first = make_uint4(0, 0, 0, 0);
  if (v0 < nvec) first = ld_stream_u4(row + v0);
  token_rank_rows(rank_slot_of, t, R, s_rank, s_row, &s_n);
  const int n = s_n;
  for (int v = v0; v < nvec; v += vec_stride()) {
    const uint4 r = v == v0 ? first : ld_stream_u4(row + v);
    for (int i = 0; i < n; ++i) rank_x[int64_t(s_row[i]) * nvec + v] = r;
  }
  if (blockIdx.y != 0) return;
  // local expert ids (expert - r * E/R) on the row's rank, -1 elsewhere
  const int Eg = E / R;
  for (int j = tid; j < n * K; j += blockDim.x) {
    const int i = j / K, k = j - i * K;
    const int r = s_rank[i];
    const int64_t e = topk_idx[int64_t(t) * K + k];
    const bool on = e >= 0 && e < E && e / Eg == r;
    rank_topk_idx[int64_t(s_row[i]) * K + k] = on ? int32_t(e - int64_t(r) * Eg) : -1;
    if (rank_topk_w != nullptr)
      rank_topk_w[int64_t(s_row[i]) * K + k] = on && w != nullptr ? w[int64_t(t) * K + k] : 0.0f;
  }
}

// Rows loaded together per thread (one batch of 16-byte loads in flight).
constexpr int kRankBatch = 8;

// ---------------------------------------------------------------------------
// expand: expert rows from rank rows
// ---------------------------------------------------------------------------
// Each CTA takes kExpandTokens consecutive tokens (and its share of their
// rows), so that one short preamble -- the tokens' routes and rank rows --
// serves several rows' streams.  Each of a token's rank rows is read once;
// its vector is stored to every expert slot that the row feeds (the experts
// of that rank): bit k of s_kmask[g][i] is set when the token's k-th
// selection goes to an expert of rank s_rank[g][i].
constexpr int kExpandTokens = 4;

__global__ void __launch_bounds__(512)
    expand_kernel(const uint4* __restrict__ rank_x,
                  const float* __restrict__ rank_topk_w,
                  const int64_t* __restrict__ topk_idx,
                  const int32_t* __restrict__ slot_of,
                  const int32_t* __restrict__ rank_slot_of, int T, int nvec, int K,
                  int E, int R, uint4* __restrict__ recv_x,
                  float* __restrict__ recv_w) {
  constexpr int G = kExpandTokens;
  __shared__ int32_t s_rk[G][32], s_dst[G][32];
  __shared__ int32_t s_rank[G][32], s_row[G][32];
  __shared__ uint32_t s_kmask[G][32];
  __shared__ int s_n[G];
  const int t0 = blockIdx.x * G;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
  pdl_wait();
  for (int j = tid; j < G * K; j += blockDim.x) {
    const int g = j / K, k = j - g * K;
    const int t = t0 + g;
    int64_t e = -1;
    int s = -1;
    if (t < T) {
      e = topk_idx[int64_t(t) * K + k];
      s = slot_of[int64_t(t) * K + k];
    }
    s_rk[g][k] = (e >= 0 && e < E && s >= 0) ? int(e / (E / R)) : -1;
    s_dst[g][k] = s;
  }
  for (int g = warp; g < G; g += nwarps) {
    if (t0 + g < T) {
      warp_rank_rows(rank_slot_of, t0 + g, R, s_rank[g], s_row[g], &s_n[g]);
    } else if (lane == 0) {
      s_n[g] = 0;
    }
  }
  __syncthreads();
  for (int g = warp; g < G; g += nwarps) {
    const int i = lane;
    uint32_t m = 0;
    if (i < s_n[g])
      for (int k = 0; k < K; ++k) m |= (s_rk[g][k] == s_rank[g][i] ? 1u : 0u) << k;
    s_kmask[g][i] = m;
  }
  __syncthreads();
#pragma unroll 1
  for (int g = 0; g < G; ++g) {
    const int n = s_n[g];
    for (int v = first_vec(); v < nvec; v += vec_stride()) {
      for (int ib = 0; ib < n; ib += kRankBatch) {
        uint4 r[kRankBatch];
#pragma unroll
        for (int j = 0; j < kRankBatch; ++j)
          r[j] = ib + j < n ? ld_stream_u4(rank_x + int64_t(s_row[g][ib + j]) * nvec + v)
                            : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < kRankBatch; ++j) {
          if (ib + j >= n) break;
          for (uint32_t m = s_kmask[g][ib + j]; m != 0; m &= m - 1)
            recv_x[int64_t(s_dst[g][__ffs(m) - 1]) * nvec + v] = r[j];
        }
      }
    }
  }
  // gate weights: lane i of warp g copies those of token g's rank row i
  if (blockIdx.y == 0 && recv_w != nullptr && rank_topk_w != nullptr)
    for (int g = warp; g < G; g += nwarps)
      if (lane < s_n[g])
        for (uint32_t m = s_kmask[g][lane]; m != 0; m &= m - 1) {
          const int k = __ffs(m) - 1;
          recv_w[s_dst[g][k]] = rank_topk_w[int64_t(s_row[g][lane]) * K + k];
        }
}

// ---------------------------------------------------------------------------
// reduce to ranks: one bf16 partial row per (token, rank)
// ---------------------------------------------------------------------------
// rank_y[row(t,r), i] = bf16( fold over k ascending with rank(e_k) = r of
// fmaf(w[t,k], Y[slot_of[t,k], i], acc) ), acc from +0 -- the destination
// rank's partial sum before sending back; the bf16 rounding of this partial
// is the extra rounding of a multi-stage reduction ("Combine: reverse
// routing plus reduction", the 256 + 1 - 256 case).
//
// The token's used selections are put in fold order -- grouped by rank
// (ranks ascending), k ascending within a group -- so that one running sum
// walks the positions p and is stored and cleared where a group ends: every
// loaded row is folded once, right after its batch arrives.  (A rank row
// always has at least one used selection in a valid layout.)
__global__ void __launch_bounds__(256)
    reduce_ranks_kernel(const uint4* __restrict__ Y, const float* __restrict__ w,
                        const int64_t* __restrict__ topk_idx,
                        const int32_t* __restrict__ slot_of,
                        const int32_t* __restrict__ rank_slot_of, int nvec,
                        int K, int E, int R, uint4* __restrict__ rank_y) {
  __shared__ int32_t s_slot[32], s_rk[32];
  __shared__ float s_w[32];
  __shared__ int32_t s_rank[32], s_row[32];
  __shared__ int32_t s_pslot[32], s_pend[32];   // per fold position
  __shared__ float s_pw[32];
  __shared__ int s_n, s_cnt;
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  pdl_wait();
  if (tid < K) {
    const int64_t e = topk_idx[int64_t(t) * K + tid];
    const int s = slot_of[int64_t(t) * K + tid];
    const bool ok = e >= 0 && e < E && s >= 0;
    s_slot[tid] = s;
    s_rk[tid] = ok ? int(e / (E / R)) : -1;
    s_w[tid] = w != nullptr ? w[int64_t(t) * K + tid] : 1.0f;
  }
  token_rank_rows(rank_slot_of, t, R, s_rank, s_row, &s_n);
  if (tid < 32) {
    // lane i: the selections of rank row i, placed after those of rows < i
    const int i = tid;
    const int n = s_n;
    uint32_t m = 0;
    if (i < n)
      for (int k = 0; k < K; ++k) m |= (s_rk[k] == s_rank[i] ? 1u : 0u) << k;
    const int c = __popc(m);
    int incl = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, d);
      if (i >= d) incl += y;
    }
    int p = incl - c;
    for (; m != 0; m &= m - 1, ++p) {
      const int k = __ffs(m) - 1;
      s_pslot[p] = s_slot[k];
      s_pw[p] = s_w[k];
      s_pend[p] = (m & (m - 1)) == 0 ? s_row[i] : -1;
    }
    if (i == 31) s_cnt = incl;
  }
  __syncthreads();
  const int cnt = s_cnt;
  for (int v = first_vec(); v < nvec; v += vec_stride()) {
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
    for (int pb = 0; pb < cnt; pb += kRankBatch) {
      uint4 r[kRankBatch];
#pragma unroll
      for (int j = 0; j < kRankBatch; ++j)
        r[j] = pb + j < cnt ? ld_stream_u4(Y + int64_t(s_pslot[pb + j]) * nvec + v)
                            : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < kRankBatch; ++j) {
        const int p = pb + j;
        if (p >= cnt) break;
        const float wk = s_pw[p];
        acc[0] = fmaf(wk, bf16_lo(r[j].x), acc[0]);
        acc[1] = fmaf(wk, bf16_hi(r[j].x), acc[1]);
        acc[2] = fmaf(wk, bf16_lo(r[j].y), acc[2]);
        acc[3] = fmaf(wk, bf16_hi(r[j].y), acc[3]);
        acc[4] = fmaf(wk, bf16_lo(r[j].z), acc[4]);
        acc[5] = fmaf(wk, bf16_hi(r[j].z), acc[5]);
        acc[6] = fmaf(wk, bf16_lo(r[j].w), acc[6]);
        acc[7] = fmaf(wk, bf16_hi(r[j].w), acc[7]);
        const int end = s_pend[p];
        if (end >= 0) {
          uint4 o;
          o.x = pack_bf16x2(acc[0], acc[1]);
          o.y = pack_bf16x2(acc[2], acc[3]);
          o.z = pack_bf16x2(acc[4], acc[5]);
          o.w = pack_bf16x2(acc[6], acc[7]);
          rank_y[int64_t(end) * nvec + v] = o;
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
        }
      }
    }
  }
}

cudaError_t launch_ranks(const RankArgs& a, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  const int nvec = a.H / 8;
  dim3 block;
  int parts;
  switch (a.op) {
    case RankArgs::kDispatch:
      split_row(nvec, 512, &block, &parts);
      return launch_pdl(dispatch_ranks_kernel, dim3(a.T, parts), block, 0, stream,
                        static_cast<const uint4*>(a.src), a.topk_idx, a.weights,
                        a.rank_slot_of, nvec, a.K, a.E, a.R, static_cast<uint4*>(a.dst),
                        a.rank_topk_idx, a.rank_topk_w);
    case RankArgs::kExpand:
      split_row(nvec, 512, &block, &parts);
      return launch_pdl(expand_kernel,
                        dim3((a.T + kExpandTokens - 1) / kExpandTokens, parts), block, 0,
                        stream, static_cast<const uint4*>(a.src), a.rank_topk_w, a.topk_idx,
                        a.slot_of, a.rank_slot_of, a.T, nvec, a.K, a.E, a.R,
                        static_cast<uint4*>(a.dst), a.recv_w);
    case RankArgs::kReduce: {
      // about seven vectors per thread: a long enough stream per CTA to
      // cover its preamble, with one CTA per token at H = 7168
      split_row(nvec, 128, &block, &parts);
      const int per_cta = parts <= 7 ? 1 : (parts + 6) / 7;
      return launch_pdl(reduce_ranks_kernel, dim3(a.T, per_cta), block, 0, stream,
                        static_cast<const uint4*>(a.src), a.weights, a.topk_idx, a.slot_of,
                        a.rank_slot_of, nvec, a.K, a.E, a.R, static_cast<uint4*>(a.dst));
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace ep

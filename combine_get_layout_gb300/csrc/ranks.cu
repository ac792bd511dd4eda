// Non-expanded (destination-major) stage ("Deep Dive - DeepEP": "Why expert
// parallelism needs a communication layer" -- a token travels once to each
// selected destination rank and an optional expansion then makes one slot
// per expert; "Dispatch: layout, move, and epilogue" -- in non-expanded
// mode a received row is a source token with its top-k metadata; "GPU
// Microarchitecture: DeepEP from First Principles" 2.1 -- receive buffer ->
// expert buffer, 1.2 -- expert-major -> destination-major -> token-major).
//
// The rank rows come from the layout (rank_slot_of, token order within each
// rank).  All kernels: one CTA per token, 16-byte vectors, bf16 rows.
#include "ep_device.cuh"
#include "ep_internal.h"

namespace ep {

// The token's destination ranks in ascending order, compacted by warp 0:
// s_rank[i], s_row[i] for i < *s_n (a token reaches at most min(K, R) <= 32
// ranks).  All threads of the block call; the block is synchronised after.
__device__ __forceinline__ void token_rank_rows(const int32_t* __restrict__ rank_slot_of,
                                                int t, int R, int32_t* s_rank,
                                                int32_t* s_row, int* s_n) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
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
  __syncthreads();
}

// ---------------------------------------------------------------------------
// dispatch to ranks: rank_x[row(t, r)] = x[t] and the row's top-k metadata
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
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
  pdl_launch_dependents();
  const uint4* row = x + int64_t(t) * nvec;
  uint4 first = make_uint4(0, 0, 0, 0);
  if (tid < nvec) first = ld_stream_u4(row + tid);
  token_rank_rows(rank_slot_of, t, R, s_rank, s_row, &s_n);
  const int n = s_n;
  const int Eg = E / R;
  // local expert ids (expert - r * E/R) on the row's rank, -1 elsewhere
  for (int j = tid; j < n * K; j += blockDim.x) {
    const int i = j / K, k = j - i * K;
    const int r = s_rank[i];
    const int64_t e = topk_idx[int64_t(t) * K + k];
    const bool on = e >= 0 && e < E && e / Eg == r;
    rank_topk_idx[int64_t(s_row[i]) * K + k] = on ? int32_t(e - int64_t(r) * Eg) : -1;
    if (rank_topk_w != nullptr)
      rank_topk_w[int64_t(s_row[i]) * K + k] = on && w != nullptr ? w[int64_t(t) * K + k] : 0.0f;
  }
  for (int v = tid; v < nvec; v += blockDim.x) {
    const uint4 r = v == tid ? first : ld_stream_u4(row + v);
    for (int i = 0; i < n; ++i) rank_x[int64_t(s_row[i]) * nvec + v] = r;
  }
}

// ---------------------------------------------------------------------------
// expand: expert rows from rank rows
// ---------------------------------------------------------------------------
constexpr int kRankBatch = 8;

__global__ void __launch_bounds__(1024)
    expand_kernel(const uint4* __restrict__ rank_x,
                  const float* __restrict__ rank_topk_w,
                  const int64_t* __restrict__ topk_idx,
                  const int32_t* __restrict__ slot_of,
                  const int32_t* __restrict__ rank_slot_of, int nvec, int K,
                  int E, int R, uint4* __restrict__ recv_x,
                  float* __restrict__ recv_w) {
  __shared__ int32_t s_src[32], s_dst[32];
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  if (tid < K) {
    const int64_t e = topk_idx[int64_t(t) * K + tid];
    const int s = slot_of[int64_t(t) * K + tid];
    const int src = (e >= 0 && e < E && s >= 0)
                        ? rank_slot_of[int64_t(t) * R + int(e / (E / R))]
                        : -1;
    s_src[tid] = src;
    s_dst[tid] = src >= 0 ? s : -1;
    if (src >= 0 && recv_w != nullptr && rank_topk_w != nullptr)
      recv_w[s] = rank_topk_w[int64_t(src) * K + tid];
  }
  __syncthreads();
  for (int v = tid; v < nvec; v += blockDim.x) {
    for (int kb = 0; kb < K; kb += kRankBatch) {
      uint4 r[kRankBatch];
#pragma unroll
      for (int j = 0; j < kRankBatch; ++j) {
        const int k = kb + j;
        const int src = k < K ? s_src[k] : -1;
        r[j] = src >= 0 ? ld_stream_u4(rank_x + int64_t(src) * nvec + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < kRankBatch; ++j) {
        const int k = kb + j;
        if (k < K && s_dst[k] >= 0) recv_x[int64_t(s_dst[k]) * nvec + v] = r[j];
      }
    }
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
__global__ void __launch_bounds__(256)
    reduce_ranks_kernel(const uint4* __restrict__ Y, const float* __restrict__ w,
                        const int64_t* __restrict__ topk_idx,
                        const int32_t* __restrict__ slot_of,
                        const int32_t* __restrict__ rank_slot_of, int nvec,
                        int K, int E, int R, uint4* __restrict__ rank_y) {
  __shared__ int32_t s_slot[32], s_rk[32];
  __shared__ float s_w[32];
  __shared__ int32_t s_rank[32], s_row[32];
  __shared__ int s_n;
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  if (tid < K) {
    const int64_t e = topk_idx[int64_t(t) * K + tid];
    const int s = slot_of[int64_t(t) * K + tid];
    const bool ok = e >= 0 && e < E && s >= 0;
    s_slot[tid] = ok ? s : -1;
    s_rk[tid] = ok ? int(e / (E / R)) : -1;
    s_w[tid] = w != nullptr ? w[int64_t(t) * K + tid] : 1.0f;
  }
  token_rank_rows(rank_slot_of, t, R, s_rank, s_row, &s_n);
  const int n = s_n;
  for (int v = tid; v < nvec; v += blockDim.x) {
    for (int i = 0; i < n; ++i) {
      const int rk = s_rank[i];
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
      for (int kb = 0; kb < K; kb += kRankBatch) {
        uint4 r[kRankBatch];
#pragma unroll
        for (int j = 0; j < kRankBatch; ++j) {
          const int k = kb + j;
          const bool use = k < K && s_rk[k] == rk;
          r[j] = use ? ld_stream_u4(Y + int64_t(s_slot[k]) * nvec + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < kRankBatch; ++j) {
          const int k = kb + j;
          if (k >= K || s_rk[k] != rk) continue;
          const float wk = s_w[k];
          acc[0] = fmaf(wk, bf16_lo(r[j].x), acc[0]);
          acc[1] = fmaf(wk, bf16_hi(r[j].x), acc[1]);
          acc[2] = fmaf(wk, bf16_lo(r[j].y), acc[2]);
          acc[3] = fmaf(wk, bf16_hi(r[j].y), acc[3]);
          acc[4] = fmaf(wk, bf16_lo(r[j].z), acc[4]);
          acc[5] = fmaf(wk, bf16_hi(r[j].z), acc[5]);
          acc[6] = fmaf(wk, bf16_lo(r[j].w), acc[6]);
          acc[7] = fmaf(wk, bf16_hi(r[j].w), acc[7]);
        }
      }
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      rank_y[int64_t(s_row[i]) * nvec + v] = o;
    }
  }
}

static int threads_for_vecs(int nvec, int cap) {
  return nvec < cap ? ((nvec + 31) / 32) * 32 : cap;
}

cudaError_t launch_ranks(const RankArgs& a, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  const int nvec = a.H / 8;
  switch (a.op) {
    case RankArgs::kDispatch:
      return launch_pdl(dispatch_ranks_kernel, dim3(a.T), dim3(threads_for_vecs(nvec, 1024)),
                        0, stream, static_cast<const uint4*>(a.src), a.topk_idx,
                        a.weights, a.rank_slot_of, nvec, a.K, a.E, a.R,
                        static_cast<uint4*>(a.dst), a.rank_topk_idx, a.rank_topk_w);
    case RankArgs::kExpand:
      return launch_pdl(expand_kernel, dim3(a.T), dim3(threads_for_vecs(nvec, 1024)), 0,
                        stream, static_cast<const uint4*>(a.src), a.rank_topk_w,
                        a.topk_idx, a.slot_of, a.rank_slot_of, nvec, a.K, a.E, a.R,
                        static_cast<uint4*>(a.dst), a.recv_w);
    case RankArgs::kReduce:
      return launch_pdl(reduce_ranks_kernel, dim3(a.T), dim3(threads_for_vecs(nvec, 128)),
                        0, stream, static_cast<const uint4*>(a.src), a.weights,
                        a.topk_idx, a.slot_of, a.rank_slot_of, nvec, a.K, a.E, a.R,
                        static_cast<uint4*>(a.dst));
  }
  return cudaErrorInvalidValue;
}

}  // namespace ep

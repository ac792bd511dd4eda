// Combine: expert-major rows -> token-major rows with the gate weights
// applied exactly once ("GPU Microarchitecture: DeepEP from First
// Principles", 1.2: Output(T0) = 0.73 x Expert2(T0) + 0.27 x Expert7(T0);
// "Deep Dive - DeepEP", "Combine: reverse routing plus reduction": fp32
// accumulation and a single final bf16 cast, so that no bf16 subtotal loses
// a small term).
//
// One CTA per token (or per slice of a token's row when tokens are few).
// Each thread owns 8 channels (one 16-byte vector) at a time, issues the loads of all of the token's selected rows for that
// vector together (up to 8 x 16 bytes in flight per thread), then folds
// them in ascending k with fmaf, acc starting at +0.0f, and stores one
// 16-byte vector of bf16 rounded to nearest even.
#include "ep_device.cuh"
#include "ep_internal.h"

namespace ep {

constexpr int kCombineKBatch = 8;

// NB: number of bf16 bias tensors added after the fold (0, 1 or 2), each in
// fp32 and in order ("Deep Dive - DeepEP", "Combine: reverse routing plus
// reduction": zero, one or two bias tensors in the combine epilogue).
// combined_w (optional): the gate weight of each (t, k) read back from its
// expert row (recv_w), 0 for an unused selection.
template <int NB>
__global__ void __launch_bounds__(256)
    combine_kernel(const uint4* __restrict__ Y, const float* __restrict__ w,
                   const int32_t* __restrict__ slot_of, int H, int K,
                   int slices, const uint4* __restrict__ b0,
                   const uint4* __restrict__ b1,
                   const float* __restrict__ recv_w,
                   float* __restrict__ combined_w, uint4* __restrict__ y) {
  // the token's used selections, compacted in ascending k
  __shared__ int32_t s_slot[kCombineMaxSlots];
  __shared__ float s_w[kCombineMaxSlots];
  __shared__ int s_cnt;
  // CTA = (token, slice of the row): few tokens still fill the GPU.
  const int t = blockIdx.x / slices;
  const int slice = blockIdx.x - t * slices;
  const int tid = threadIdx.x;
  const int nvec = H >> 3;
  const int per = (nvec + slices - 1) / slices;
  const int v0 = slice * per, v1 = min(nvec, v0 + per);
  pdl_wait();
  if (tid < 32) {
    // warp 0 reads the route and compacts the used selections (a sparse
    // route -- e.g. a token's few ranks out of many -- then costs one batch
    // of loads, not one per group of eight entries)
    const uint32_t lt = lanemask_lt();
    int n = 0;
    for (int c0 = 0; c0 < K; c0 += 32) {
      const int k = c0 + tid;
      const int sl = k < K ? slot_of[int64_t(t) * K + k] : -1;
      const float wk = k < K && w != nullptr ? w[int64_t(t) * K + k] : 1.0f;
      const uint32_t m = __ballot_sync(0xffffffffu, sl >= 0);
      if (sl >= 0) {
        const int pos = n + __popc(m & lt);
        s_slot[pos] = sl;
        s_w[pos] = wk;
      }
      if (k < K && combined_w != nullptr && slice == 0)
        combined_w[int64_t(t) * K + k] = sl >= 0 ? recv_w[sl] : 0.0f;
      n += __popc(m);
    }
    if (tid == 0) s_cnt = n;
  }
  __syncthreads();
  const int cnt = s_cnt;

  for (int v = v0 + tid; v < v1; v += blockDim.x) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (int kb = 0; kb < cnt; kb += kCombineKBatch) {
      uint4 r[kCombineKBatch];
#pragma unroll
      for (int j = 0; j < kCombineKBatch; ++j)
        r[j] = kb + j < cnt ? ld_stream_u4(Y + int64_t(s_slot[kb + j]) * nvec + v)
                            : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < kCombineKBatch; ++j) {
        if (kb + j >= cnt) break;
        const float wk = s_w[kb + j];
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
    if (NB >= 1) {
      const uint4 b = ld_stream_u4(b0 + int64_t(t) * nvec + v);
      acc[0] += bf16_lo(b.x); acc[1] += bf16_hi(b.x);
      acc[2] += bf16_lo(b.y); acc[3] += bf16_hi(b.y);
      acc[4] += bf16_lo(b.z); acc[5] += bf16_hi(b.z);
      acc[6] += bf16_lo(b.w); acc[7] += bf16_hi(b.w);
    }
    if (NB >= 2) {
      const uint4 b = ld_stream_u4(b1 + int64_t(t) * nvec + v);
      acc[0] += bf16_lo(b.x); acc[1] += bf16_hi(b.x);
      acc[2] += bf16_lo(b.y); acc[3] += bf16_hi(b.y);
      acc[4] += bf16_lo(b.z); acc[5] += bf16_hi(b.z);
      acc[6] += bf16_lo(b.w); acc[7] += bf16_hi(b.w);
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    y[int64_t(t) * nvec + v] = o;
  }
}

// CTAs wanted in flight before rows are split across CTAs.
constexpr int kCombineMinCtas = 8192;

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  const int nvec = a.H / 8;
  const int threads = nvec >= 128 ? 128 : ((nvec + 31) / 32) * 32;
  // Split each row into slices of at least `threads` vectors when there are
  // too few tokens to keep the GPU's memory system busy.
  int slices = 1;
  if (a.T < kCombineMinCtas) {
    slices = (kCombineMinCtas + a.T - 1) / a.T;
    const int max_slices = (nvec + threads - 1) / threads;
    if (slices > max_slices) slices = max_slices;
  }
  // Biases in the order given; a single one always goes in the first slot.
  const uint4* b0 = static_cast<const uint4*>(a.bias0 != nullptr ? a.bias0 : a.bias1);
  const uint4* b1 = static_cast<const uint4*>(a.bias0 != nullptr ? a.bias1 : nullptr);
  const int nb = (b0 != nullptr) + (b1 != nullptr);
  const dim3 grid(a.T * slices), block(threads);
  const uint4* Y = static_cast<const uint4*>(a.expert_out);
  uint4* y = static_cast<uint4*>(a.y);
  if (nb == 0)
    return launch_ex(a.pdl, combine_kernel<0>, grid, block, 0, stream, Y, a.topk_weights,
                     a.slot_of, a.H, a.K, slices, b0, b1, a.recv_w, a.combined_w, y);
  if (nb == 1)
    return launch_ex(a.pdl, combine_kernel<1>, grid, block, 0, stream, Y, a.topk_weights,
                     a.slot_of, a.H, a.K, slices, b0, b1, a.recv_w, a.combined_w, y);
  return launch_ex(a.pdl, combine_kernel<2>, grid, block, 0, stream, Y, a.topk_weights,
                   a.slot_of, a.H, a.K, slices, b0, b1, a.recv_w, a.combined_w, y);
}

// ---------------------------------------------------------------------------
// combine backward
// ---------------------------------------------------------------------------
// For y[t] = sum_k w[t,k] * Y[slot_of[t,k]] ("Deep Dive - DeepEP", combine
// section, backward duality -- the transpose of the weighted row sum, plus
// the gate gradient):
//   grad_Y[slot, i] = bf16( w[t,k] * dy[t,i] )   (fp32 product, one rounding)
//   grad_w[t,k]     = sum_i dy[t,i] * Y[slot, i] (fp32, fixed order: each
//                     thread folds its vectors, then a warp tree, then the
//                     warps in order)
// One CTA per token; KB bounds the number of selections held in registers.
template <int KB, bool kGradW>
__global__ void __launch_bounds__(256)
    combine_backward_kernel(const uint4* __restrict__ dy,
                            const float* __restrict__ w,
                            const int32_t* __restrict__ slot_of,
                            const uint4* __restrict__ Y, int H, int K,
                            uint4* __restrict__ grad_Y,
                            float* __restrict__ grad_w) {
  __shared__ int32_t s_slot[32];
  __shared__ float s_w[32];
  __shared__ float s_red[8][KB];
  const int t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nvec = H >> 3;
  pdl_wait();
  if (tid < K) {
    s_slot[tid] = slot_of[int64_t(t) * K + tid];
    s_w[tid] = w != nullptr ? w[int64_t(t) * K + tid] : 1.0f;
  }
  __syncthreads();

  float part[KB];
#pragma unroll
  for (int k = 0; k < KB; ++k) part[k] = 0.0f;
  for (int v = tid; v < nvec; v += blockDim.x) {
    const uint4 g = ld_stream_u4(dy + int64_t(t) * nvec + v);
    const float gf[8] = {bf16_lo(g.x), bf16_hi(g.x), bf16_lo(g.y), bf16_hi(g.y),
                         bf16_lo(g.z), bf16_hi(g.z), bf16_lo(g.w), bf16_hi(g.w)};
#pragma unroll
    for (int kb = 0; kb < KB; kb += kCombineKBatch) {
      if (kb >= K) break;
      // the batch's expert rows are loaded together, then used
      uint4 r[kCombineKBatch];
      if (kGradW) {
#pragma unroll
        for (int j = 0; j < kCombineKBatch; ++j) {
          const int k = kb + j;
          const int sl = k < K ? s_slot[k] : -1;
          r[j] = sl >= 0 ? ld_stream_u4(Y + int64_t(sl) * nvec + v) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int j = 0; j < kCombineKBatch; ++j) {
        const int k = kb + j;
        if (k >= K) break;
        const int sl = s_slot[k];
        if (sl < 0) continue;
        const float wk = s_w[k];
        uint4 o;
        o.x = pack_bf16x2(wk * gf[0], wk * gf[1]);
        o.y = pack_bf16x2(wk * gf[2], wk * gf[3]);
        o.z = pack_bf16x2(wk * gf[4], wk * gf[5]);
        o.w = pack_bf16x2(wk * gf[6], wk * gf[7]);
        grad_Y[int64_t(sl) * nvec + v] = o;
        if (kGradW) {
          float p = part[k];
          p = fmaf(gf[0], bf16_lo(r[j].x), p);
          p = fmaf(gf[1], bf16_hi(r[j].x), p);
          p = fmaf(gf[2], bf16_lo(r[j].y), p);
          p = fmaf(gf[3], bf16_hi(r[j].y), p);
          p = fmaf(gf[4], bf16_lo(r[j].z), p);
          p = fmaf(gf[5], bf16_hi(r[j].z), p);
          p = fmaf(gf[6], bf16_lo(r[j].w), p);
          p = fmaf(gf[7], bf16_hi(r[j].w), p);
          part[k] = p;
        }
      }
    }
  }
  if (kGradW) {
#pragma unroll
    for (int k = 0; k < KB; ++k) {
      float p = part[k];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
      if (lane == 0) s_red[warp][k] = p;
    }
    __syncthreads();
    if (tid < K) {
      float acc = 0.0f;
      for (int wi = 0; wi < (int)(blockDim.x >> 5); ++wi) acc += s_red[wi][tid];
      grad_w[int64_t(t) * K + tid] = s_slot[tid] >= 0 ? acc : 0.0f;
    }
  }
}

cudaError_t launch_combine_backward(const CombineBackwardArgs& a, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  const int nvec = a.H / 8;
  const int threads = nvec >= 256 ? 256 : ((nvec + 31) / 32) * 32;
  const uint4* dy = static_cast<const uint4*>(a.dy);
  const uint4* Y = static_cast<const uint4*>(a.expert_out);
  uint4* gY = static_cast<uint4*>(a.grad_expert_out);
  const dim3 grid(a.T), block(threads);
  const bool gw = a.grad_w != nullptr;
  if (a.K <= 8) {
    auto kern = gw ? combine_backward_kernel<8, true> : combine_backward_kernel<8, false>;
    return launch_pdl(kern, grid, block, 0, stream, dy, a.topk_weights, a.slot_of, Y,
                      a.H, a.K, gY, a.grad_w);
  }
  auto kern = gw ? combine_backward_kernel<32, true> : combine_backward_kernel<32, false>;
  return launch_pdl(kern, grid, block, 0, stream, dy, a.topk_weights, a.slot_of, Y,
                    a.H, a.K, gY, a.grad_w);
}

}  // namespace ep

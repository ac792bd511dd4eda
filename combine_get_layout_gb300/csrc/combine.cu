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

__global__ void __launch_bounds__(256)
    combine_kernel(const uint4* __restrict__ Y, const float* __restrict__ w,
                   const int32_t* __restrict__ slot_of, int H, int K,
                   int slices, uint4* __restrict__ y) {
  __shared__ int32_t s_slot[32];
  __shared__ float s_w[32];
  // CTA = (token, slice of the row): few tokens still fill the GPU.
  const int t = blockIdx.x / slices;
  const int slice = blockIdx.x - t * slices;
  const int tid = threadIdx.x;
  const int nvec = H >> 3;
  const int per = (nvec + slices - 1) / slices;
  const int v0 = slice * per, v1 = min(nvec, v0 + per);
  pdl_wait();
  pdl_launch_dependents();
  if (tid < K) {
    s_slot[tid] = slot_of[int64_t(t) * K + tid];
    s_w[tid] = w != nullptr ? w[int64_t(t) * K + tid] : 1.0f;
  }
  __syncthreads();

  for (int v = v0 + tid; v < v1; v += blockDim.x) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (int kb = 0; kb < K; kb += kCombineKBatch) {
      uint4 r[kCombineKBatch];
#pragma unroll
      for (int j = 0; j < kCombineKBatch; ++j) {
        const int k = kb + j;
        const int sl = k < K ? s_slot[k] : -1;
        r[j] = sl >= 0 ? ld_stream_u4(Y + int64_t(sl) * nvec + v)
                       : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < kCombineKBatch; ++j) {
        const int k = kb + j;
        if (k >= K || s_slot[k] < 0) continue;
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
    y[int64_t(t) * nvec + v] = o;
  }
}

// CTAs wanted in flight before rows are split across CTAs.
constexpr int kCombineMinCtas = 2048;

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
  return launch_pdl(combine_kernel, dim3(a.T * slices), dim3(threads), 0, stream,
                    static_cast<const uint4*>(a.expert_out), a.topk_weights,
                    a.slot_of, a.H, a.K, slices, static_cast<uint4*>(a.y));
}

}  // namespace ep

// Dispatch, expanded mode: token-major rows -> expert-major rows
// ("GPU Microarchitecture: DeepEP from First Principles", 1.1; "Deep Dive -
// DeepEP", "Dispatch: layout, move, and epilogue").  Every unmasked (t, k)
// receives a copy of x[t] at row slot_of[t, k]; its gate weight rides along
// in recv_w.  Destination ranks are row ranges of the same buffer, so the
// destination-major and expert-major stages are one scatter.  x is read
// once and every destination row written once: the algorithmic bytes.
// FP8 rows follow "Precision: FP8 on the wire, BF16 for the reduction": one
// fp32 scale per 128 channels, quantised once per token and written to each
// of its rows.
#include "ep_device.cuh"
#include "ep_internal.h"
#include "fp8_quant.cuh"

namespace ep {

// ---------------------------------------------------------------------------
// bf16: bit copies with 16-byte vectors
// ---------------------------------------------------------------------------
// One CTA per token, or two when the row has more than 512 vectors (two
// smaller CTAs per SM slot overlap one's route read with the other's
// stream); each thread owns one 16-byte vector of the row at a time (8
// channels): one load, then one store per selected expert.  The first load is
// issued before the route is read, so the two latencies overlap.  (A variant
// that staged whole rows in shared memory through a ring of bulk copies --
// one load and K bulk stores per token -- measured ~10% slower on GB300 at
// the DeepSeek-V3 prefill shape: the register path keeps more stores in
// flight per SM.)
__global__ void __launch_bounds__(512)
    dispatch_bf16_kernel(const uint4* __restrict__ x,
                         const float* __restrict__ w,
                         const int32_t* __restrict__ slot_of, int nvec, int K,
                         uint4* __restrict__ recv_x,
                         float* __restrict__ recv_w) {
  __shared__ int32_t s_slot[32];
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  pdl_wait();
  const uint4* row = x + int64_t(t) * nvec;
  const int v0 = first_vec();
  uint4 first = make_uint4(0, 0, 0, 0);
  if (v0 < nvec) first = ld_stream_u4(row + v0);
  if (tid < K) {
    const int sl = slot_of[int64_t(t) * K + tid];
    s_slot[tid] = sl;
    if (sl >= 0 && w != nullptr && recv_w != nullptr && blockIdx.y == 0)
      recv_w[sl] = w[int64_t(t) * K + tid];
  }
  __syncthreads();
  for (int v = v0; v < nvec; v += vec_stride()) {
    const uint4 r = v == v0 ? first : ld_stream_u4(row + v);
    for (int k = 0; k < K; ++k) {
      const int sl = s_slot[k];
      if (sl >= 0) recv_x[int64_t(sl) * nvec + v] = r;
    }
  }
}

// ---------------------------------------------------------------------------
// FP8 E4M3 with 1x128 scales
// ---------------------------------------------------------------------------
// Where the scale of (row, block) lives: row-major [cap, H/128], or
// column-major [H/128, ld] with ld = cap rounded up to 4 (the layout for TMA
// consumers: each block's scales are one 16-byte-aligned column).
template <bool kColMajor>
__device__ __forceinline__ int64_t scale_index(int64_t row, int blk, int nblk, int64_t ld) {
  return kColMajor ? int64_t(blk) * ld + row : row * nblk + blk;
}

// One CTA per token; thread u owns 16 consecutive channels (two 16-byte
// loads), so 8 lanes cover one 128-channel block: exact amax by three
// shuffles, scale = amax / 448, 16 E4M3 bytes written with one 16-byte store
// per selected expert, and the block's scale by the group's first lane.
// kWide: x is 32-byte aligned and each thread's 16 channels come in one
// 256-bit load.
template <bool kColMajor, bool kWide>
__global__ void __launch_bounds__(1024)
    dispatch_fp8_kernel(const uint4* __restrict__ x,
                        const float* __restrict__ w,
                        const int32_t* __restrict__ slot_of, int H, int K,
                        int64_t scale_ld, uint8_t* __restrict__ recv_q,
                        float* __restrict__ recv_scale,
                        float* __restrict__ recv_w) {
  __shared__ int32_t s_slot[32];
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  const int nvec = H >> 3;     // 16-byte bf16 vectors per row
  const int n16 = H >> 4;      // 16-channel groups per row
  const int nblk = H >> 7;     // 128-channel scale blocks per row
  pdl_wait();
  if (tid < K) {
    const int sl = slot_of[int64_t(t) * K + tid];
    s_slot[tid] = sl;
    if (sl >= 0 && w != nullptr && recv_w != nullptr)
      recv_w[sl] = w[int64_t(t) * K + tid];
  }
  __syncthreads();

  // blockDim is a multiple of 32, so each aligned group of 8 lanes covers
  // one whole 128-channel block.
  for (int base = 0; base < n16; base += blockDim.x) {
    const int u = base + tid;
    const bool active = u < n16;
    uint4 r0 = make_uint4(0, 0, 0, 0), r1 = r0;
    if (active) {
      const uint4* p = x + int64_t(t) * nvec + 2 * u;
      if (kWide) {
        ld_stream_u4x2(p, r0, r1);
      } else {
        r0 = ld_stream_u4(p);
        r1 = ld_stream_u4(p + 1);
      }
    }
    uint4 q;
    float scale;
    quantize_group16(r0, r1, &q, &scale);
    if (active) {
      const bool leader = (tid & 7) == 0;
      for (int k = 0; k < K; ++k) {
        const int sl = s_slot[k];
        if (sl < 0) continue;
        *reinterpret_cast<uint4*>(recv_q + int64_t(sl) * H + int64_t(u) * 16) = q;
        if (leader) recv_scale[scale_index<kColMajor>(sl, u >> 3, nblk, scale_ld)] = scale;
      }
    }
  }
}

// Pre-quantised input ("Deep Dive - DeepEP", "Precision: FP8 on the wire,
// BF16 for the reduction": FP8 values plus scale factors): bit copies of the
// token's E4M3 row (16 bytes per thread) and of its scales.
template <bool kColMajor>
__global__ void __launch_bounds__(1024)
    dispatch_fp8_copy_kernel(const uint4* __restrict__ x_q,
                             const float* __restrict__ x_scale,
                             const float* __restrict__ w,
                             const int32_t* __restrict__ slot_of, int H, int K,
                             int64_t scale_ld, uint8_t* __restrict__ recv_q,
                             float* __restrict__ recv_scale,
                             float* __restrict__ recv_w) {
  __shared__ int32_t s_slot[32];
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  const int n16 = H >> 4;      // 16-byte vectors of E4M3 per row
  const int nblk = H >> 7;
  pdl_wait();
  if (tid < K) {
    const int sl = slot_of[int64_t(t) * K + tid];
    s_slot[tid] = sl;
    if (sl >= 0 && w != nullptr && recv_w != nullptr)
      recv_w[sl] = w[int64_t(t) * K + tid];
  }
  __syncthreads();
  for (int u = tid; u < n16; u += blockDim.x) {
    const uint4 q = ld_stream_u4(x_q + int64_t(t) * n16 + u);
    for (int k = 0; k < K; ++k) {
      const int sl = s_slot[k];
      if (sl >= 0) *reinterpret_cast<uint4*>(recv_q + int64_t(sl) * H + int64_t(u) * 16) = q;
    }
  }
  for (int b = tid; b < nblk; b += blockDim.x) {
    const float sc = x_scale[int64_t(t) * nblk + b];
    for (int k = 0; k < K; ++k) {
      const int sl = s_slot[k];
      if (sl >= 0) recv_scale[scale_index<kColMajor>(sl, b, nblk, scale_ld)] = sc;
    }
  }
}

// ---------------------------------------------------------------------------
// zero the alignment gap rows [expert_end[e], expert_start[e+1])
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    zero_padding_kernel(const int32_t* __restrict__ expert_start,
                        const int32_t* __restrict__ expert_end, int E,
                        int64_t row_bytes, int scale_per_row, int64_t scale_ld,
                        uint8_t* __restrict__ recv_x,
                        float* __restrict__ recv_scale,
                        float* __restrict__ recv_w) {
  pdl_wait();
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    const int64_t s0 = expert_end[e], s1 = expert_start[e + 1];
    if (s1 <= s0) continue;
    uint4* dst = reinterpret_cast<uint4*>(recv_x + s0 * row_bytes);
    const int64_t nv = (s1 - s0) * row_bytes / 16;
    for (int64_t i = threadIdx.x; i < nv; i += blockDim.x) dst[i] = make_uint4(0, 0, 0, 0);
    if (recv_scale != nullptr && scale_ld == 0)
      for (int64_t i = s0 * scale_per_row + threadIdx.x; i < s1 * scale_per_row; i += blockDim.x)
        recv_scale[i] = 0.0f;
    if (recv_scale != nullptr && scale_ld > 0)  // column-major scales
      for (int64_t i = threadIdx.x; i < (s1 - s0) * scale_per_row; i += blockDim.x) {
        const int64_t c = i / (s1 - s0), r = s0 + (i - c * (s1 - s0));
        recv_scale[c * scale_ld + r] = 0.0f;
      }
    if (recv_w != nullptr)
      for (int64_t s = s0 + threadIdx.x; s < s1; s += blockDim.x) recv_w[s] = 0.0f;
  }
}

// Self-test of mbar_wait: the barrier expects one arrival that never comes.
__global__ void __launch_bounds__(32) wait_selftest_kernel(uint64_t timeout_ns, int32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  pdl_wait();
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, timeout_ns)) record_error(err, ERRBIT_TIMEOUT);
  }
}

cudaError_t launch_wait_selftest(uint64_t timeout_ns, int32_t* err, cudaStream_t stream) {
  return launch_pdl(wait_selftest_kernel, dim3(1), dim3(32), 0, stream, timeout_ns, err);
}

cudaError_t prepare_dispatch_kernels() { return cudaSuccess; }

// Exhaustive check of the FP8 dispatch's block quotient (BlockQuotient):
// block b takes the block maximum amax = the positive bf16 with bits b + 1
// (every finite one, then +inf), every thread a share of the 65536 bf16
// values x with |x| <= amax; counts[0] += pairs whose E4M3 codes differ from
// those of __fdiv_rn, counts[1] += pairs whose fp32 quotients differ,
// counts[2] += those of them whose IEEE quotient is a normal fp32 number;
// *first = (amax bits << 16 | x bits) of one code mismatch.
__global__ void __launch_bounds__(256)
    fp8_quotient_selftest_kernel(unsigned long long* __restrict__ counts,
                                 int32_t* __restrict__ first) {
  const uint32_t ab = blockIdx.x + 1;
  const float amax = __uint_as_float(ab << 16);
  const float s = __fdiv_rn(amax, 448.0f);
  const BlockQuotient div(s);
  unsigned long long bad_code = 0, bad_f32 = 0, bad_normal = 0;
  for (uint32_t xb = threadIdx.x; xb < 65536u; xb += blockDim.x) {
    const float x = __uint_as_float(xb << 16);
    if (!(fabsf(x) <= amax)) continue;  // also NaN
    const float qa = div(x), qb = __fdiv_rn(x, s);
    const bool differ = __float_as_uint(qa) != __float_as_uint(qb);
    bad_f32 += differ;
    bad_normal += differ && fabsf(qb) >= 0x1p-126f;
    if (pack_e4m3x2(qa, 0.0f) != pack_e4m3x2(qb, 0.0f)) {
      ++bad_code;
      atomicCAS(first, -1, int32_t((ab << 16) | xb));
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    bad_code += __shfl_xor_sync(0xffffffffu, bad_code, o);
    bad_f32 += __shfl_xor_sync(0xffffffffu, bad_f32, o);
    bad_normal += __shfl_xor_sync(0xffffffffu, bad_normal, o);
  }
  if ((threadIdx.x & 31) == 0 && (bad_code | bad_f32)) {
    atomicAdd(&counts[0], bad_code);
    atomicAdd(&counts[1], bad_f32);
    atomicAdd(&counts[2], bad_normal);
  }
}

cudaError_t launch_fp8_quotient_selftest(unsigned long long* counts, int32_t* first,
                                         cudaStream_t stream) {
  cudaError_t st = cudaMemsetAsync(counts, 0, 3 * sizeof(unsigned long long), stream);
  if (st == cudaSuccess) st = cudaMemsetAsync(first, 0xff, sizeof(int32_t), stream);
  if (st != cudaSuccess) return st;
  // positive bf16 block maxima: bits 0x0001 .. 0x7f7f (finite), 0x7f80 (+inf)
  fp8_quotient_selftest_kernel<<<0x7f80, 256, 0, stream>>>(counts, first);
  return cudaGetLastError();
}

static int threads_for(int n) { return n < 1024 ? ((n + 31) / 32) * 32 : 1024; }

cudaError_t launch_zero_padding_bf16(const int32_t* expert_start, const int32_t* expert_end,
                                     int E, int H, void* rows, cudaStream_t stream) {
  const int grid = E < 1024 ? E : 1024;
  return launch_pdl(zero_padding_kernel, dim3(grid), dim3(256), 0, stream, expert_start,
                    expert_end, E, int64_t(H) * 2, 0, int64_t(0),
                    static_cast<uint8_t*>(rows), static_cast<float*>(nullptr),
                    static_cast<float*>(nullptr));
}

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t stream) {
  cudaError_t st;
  if (a.T > 0) {
    if (!a.fp8) {
      const int nvec = a.H / 8;
      dim3 block;
      int parts;
      split_row(nvec, 512, &block, &parts);
      st = launch_ex(a.pdl, dispatch_bf16_kernel, dim3(a.T, parts), block, 0, stream,
                     static_cast<const uint4*>(a.x), a.topk_weights, a.slot_of, nvec, a.K,
                     static_cast<uint4*>(a.recv_x), a.recv_w);
    } else if (a.x_q == nullptr) {
      // rows start at multiples of 2H >= 256 bytes, so x's own alignment decides
      const bool wide = (reinterpret_cast<uintptr_t>(a.x) & 31) == 0;
      auto kern = a.scale_col_major
                      ? (wide ? dispatch_fp8_kernel<true, true> : dispatch_fp8_kernel<true, false>)
                      : (wide ? dispatch_fp8_kernel<false, true> : dispatch_fp8_kernel<false, false>);
      st = launch_ex(a.pdl, kern, dim3(a.T), dim3(threads_for(a.H / 16)), 0, stream,
                     static_cast<const uint4*>(a.x), a.topk_weights, a.slot_of, a.H,
                     a.K, a.scale_ld, static_cast<uint8_t*>(a.recv_x), a.recv_scale,
                     a.recv_w);
    } else {
      auto kern = a.scale_col_major ? dispatch_fp8_copy_kernel<true>
                                    : dispatch_fp8_copy_kernel<false>;
      st = launch_ex(a.pdl, kern, dim3(a.T), dim3(threads_for(a.H / 16)), 0, stream,
                     reinterpret_cast<const uint4*>(a.x_q), a.x_scale, a.topk_weights,
                     a.slot_of, a.H, a.K, a.scale_ld, static_cast<uint8_t*>(a.recv_x),
                     a.recv_scale, a.recv_w);
    }
    if (st != cudaSuccess) return st;
  }
  if (a.zero_padding) {
    const int64_t row_bytes = a.fp8 ? int64_t(a.H) : int64_t(a.H) * 2;
    int grid = a.E < 1024 ? a.E : 1024;
    st = launch_pdl(zero_padding_kernel, dim3(grid), dim3(256), 0, stream,
                    a.expert_start, a.expert_end, a.E, row_bytes,
                    a.fp8 ? a.H / 128 : 0, a.scale_col_major ? a.scale_ld : int64_t(0),
                    static_cast<uint8_t*>(a.recv_x), a.fp8 ? a.recv_scale : nullptr,
                    a.recv_w);
    if (st != cudaSuccess) return st;
  }
  return cudaSuccess;
}

}  // namespace ep

// Dispatch, expanded mode: token-major rows -> expert-major rows
// ("GPU Microarchitecture: DeepEP from First Principles", 1.1; "Deep Dive -
// DeepEP", "Dispatch: layout, move, and epilogue").  Every unmasked (t, k)
// receives a copy of x[t] at row slot_of[t, k]; its gate weight rides along
// in recv_w.  Destination ranks are row ranges of the same buffer, so the
// destination-major and expert-major stages are one scatter.
//
// bf16: each CTA is one warp streaming whole rows through a ring of shared
//   memory stages with bulk copies (TMA): one global->shared load per token,
//   K shared->global stores (one per selected expert).  x is read once and
//   each destination row written once: exactly the algorithmic bytes.
// FP8 ("Precision: FP8 on the wire, BF16 for the reduction"): one CTA per
//   token; each half-warp owns one 128-channel block: 16-byte loads, exact
//   amax by shuffles, scale = amax / 448, q = E4M3(x / scale) rounded to
//   nearest even and saturated, then K 8-byte stores per lane.
#include "ep_device.cuh"
#include "ep_internal.h"

namespace ep {

// ---------------------------------------------------------------------------
// bf16 rows through a bulk-copy ring
// ---------------------------------------------------------------------------
constexpr int kBarrierBytes = 128;  // stage barriers, padded to 128 bytes
constexpr int kMaxStages = 8;
constexpr int kStageBudget = 64 * 1024;  // shared-memory target per CTA

__global__ void __launch_bounds__(32)
    dispatch_bf16_kernel(const uint8_t* __restrict__ x,
                         const float* __restrict__ w,
                         const int32_t* __restrict__ slot_of, int T, int K,
                         uint32_t row_bytes, int stages,
                         uint8_t* __restrict__ recv_x,
                         float* __restrict__ recv_w, int32_t* err) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint8_t* ring = smem + kBarrierBytes;
  const int lane = threadIdx.x;
  const int n = T > static_cast<int>(blockIdx.x)
                    ? (T - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1
                    : 0;
  if (n == 0) {
    pdl_wait();
    pdl_launch_dependents();
    return;
  }

  if (lane == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  pdl_wait();
  pdl_launch_dependents();

  auto token = [&](int i) { return static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x); };
  auto issue = [&](int i) {  // lane 0 only
    const int s = i % stages;
    mbar_arrive_expect_tx(&full[s], row_bytes);
    bulk_load(ring + size_t(s) * row_bytes, x + size_t(token(i)) * row_bytes,
              row_bytes, &full[s]);
  };

  if (lane == 0)
    for (int i = 0; i < stages && i < n; ++i) issue(i);

  bool ok = true;
  int i = 0;
  for (; i < n; ++i) {
    const int t = token(i);
    const int s = i % stages;
    // route of token t, one selection per lane (K <= 32)
    int slot = -1;
    if (lane < K) {
      slot = slot_of[int64_t(t) * K + lane];
      if (slot >= 0 && w != nullptr && recv_w != nullptr)
        recv_w[slot] = w[int64_t(t) * K + lane];
    }
    // Lane 0 alone waits (only the bulk copies read the stage), so the
    // outcome is the same on every lane.
    int arrived = 0;
    if (lane == 0) arrived = mbar_wait(&full[s], (i / stages) & 1, kWaitTimeoutNs);
    if (!__shfl_sync(0xffffffffu, arrived, 0)) {
      ok = false;
      break;
    }
    for (int k = 0; k < K; ++k) {
      const int sl = __shfl_sync(0xffffffffu, slot, k);
      if (lane == 0 && sl >= 0)
        bulk_store(recv_x + size_t(sl) * row_bytes, ring + size_t(s) * row_bytes,
                   row_bytes);
    }
    if (lane == 0) {
      bulk_commit();
      // Refill the stage of the previous token once its stores have read
      // it; the stores of this token stay in flight.
      if (i >= 1 && i - 1 + stages < n) {
        bulk_wait_read<1>();
        issue(i - 1 + stages);
      }
    }
    __syncwarp();
  }

  if (!ok) {
    record_error(err, ERRBIT_TIMEOUT);
    // Drain the loads still outstanding (bounded) before leaving.
    if (lane == 0) {
      const int last = min(n, (i >= 1 ? i - 1 : 0) + stages);
      for (int j = i; j < last; ++j)
        (void)mbar_wait(&full[j % stages], (j / stages) & 1, kWaitTimeoutNs);
    }
  }
  if (lane == 0) bulk_wait_all<0>();
}

// ---------------------------------------------------------------------------
// FP8 E4M3 with 1x128 scales
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
    dispatch_fp8_kernel(const uint4* __restrict__ x,
                        const float* __restrict__ w,
                        const int32_t* __restrict__ slot_of, int T, int H,
                        int K, uint8_t* __restrict__ recv_q,
                        float* __restrict__ recv_scale,
                        float* __restrict__ recv_w) {
  __shared__ int32_t s_slot[32];
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  const int nvec = H >> 3;     // 16-byte vectors (8 channels) per row
  const int nblk = H >> 7;     // 128-channel scale blocks per row
  pdl_wait();
  pdl_launch_dependents();
  if (tid < K) {
    const int sl = slot_of[int64_t(t) * K + tid];
    s_slot[tid] = sl;
    if (sl >= 0 && w != nullptr && recv_w != nullptr)
      recv_w[sl] = w[int64_t(t) * K + tid];
  }
  __syncthreads();

  // blockDim is a multiple of 32, so the 16 lanes of a half-warp always
  // cover one whole 128-channel block.
  for (int base = 0; base < nvec; base += blockDim.x) {
    const int v = base + tid;
    const bool active = v < nvec;
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (active) raw = ld_stream_u4(x + int64_t(t) * nvec + v);
    float f[8];
    f[0] = bf16_lo(raw.x); f[1] = bf16_hi(raw.x);
    f[2] = bf16_lo(raw.y); f[3] = bf16_hi(raw.y);
    f[4] = bf16_lo(raw.z); f[5] = bf16_hi(raw.z);
    f[6] = bf16_lo(raw.w); f[7] = bf16_hi(raw.w);
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    uint2 q = make_uint2(0, 0);
    float scale = 0.0f;
    if (amax != 0.0f) {
      scale = __fdiv_rn(amax, 448.0f);
      uint16_t p[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        p[j] = pack_e4m3x2(__fdiv_rn(f[2 * j], scale), __fdiv_rn(f[2 * j + 1], scale));
      q.x = uint32_t(p[0]) | (uint32_t(p[1]) << 16);
      q.y = uint32_t(p[2]) | (uint32_t(p[3]) << 16);
    }
    if (active) {
      const int blk = v >> 4;
      const bool leader = (tid & 15) == 0;
      for (int k = 0; k < K; ++k) {
        const int sl = s_slot[k];
        if (sl < 0) continue;
        *reinterpret_cast<uint2*>(recv_q + int64_t(sl) * H + int64_t(v) * 8) = q;
        if (leader) recv_scale[int64_t(sl) * nblk + blk] = scale;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// zero the alignment gap rows [expert_end[e], expert_start[e+1])
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    zero_padding_kernel(const int32_t* __restrict__ expert_start,
                        const int32_t* __restrict__ expert_end, int E,
                        int64_t row_bytes, int scale_per_row,
                        uint8_t* __restrict__ recv_x,
                        float* __restrict__ recv_scale,
                        float* __restrict__ recv_w) {
  pdl_wait();
  pdl_launch_dependents();
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    const int64_t s0 = expert_end[e], s1 = expert_start[e + 1];
    if (s1 <= s0) continue;
    uint4* dst = reinterpret_cast<uint4*>(recv_x + s0 * row_bytes);
    const int64_t nv = (s1 - s0) * row_bytes / 16;
    for (int64_t i = threadIdx.x; i < nv; i += blockDim.x) dst[i] = make_uint4(0, 0, 0, 0);
    if (recv_scale != nullptr)
      for (int64_t i = s0 * scale_per_row + threadIdx.x; i < s1 * scale_per_row; i += blockDim.x)
        recv_scale[i] = 0.0f;
    if (recv_w != nullptr)
      for (int64_t s = s0 + threadIdx.x; s < s1; s += blockDim.x) recv_w[s] = 0.0f;
  }
}

// Self-test of mbar_wait: the barrier expects one arrival that never comes.
__global__ void __launch_bounds__(32) wait_selftest_kernel(uint64_t timeout_ns, int32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, timeout_ns)) record_error(err, ERRBIT_TIMEOUT);
  }
}

cudaError_t launch_wait_selftest(uint64_t timeout_ns, int32_t* err, cudaStream_t stream) {
  return launch_pdl(wait_selftest_kernel, dim3(1), dim3(32), 0, stream, timeout_ns, err);
}

cudaError_t prepare_dispatch_kernels() {
  return allow_max_dynamic_smem(dispatch_bf16_kernel, device_info().max_smem_optin);
}

// CTAs of the bf16 kernel resident per SM for a given shared-memory size
// (cached: the last query per thread).
static int bf16_ctas_per_sm(int smem) {
  thread_local int last_dev = -1, last_smem = -1, last_val = 1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev == last_dev && smem == last_smem) return last_val;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_bf16_kernel, 32,
                                                    smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  last_dev = dev;
  last_smem = smem;
  last_val = per_sm;
  return per_sm;
}

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t stream) {
  cudaError_t st;
  if (a.T > 0) {
    if (!a.fp8) {
      const uint32_t row_bytes = uint32_t(a.H) * 2u;
      int stages = kStageBudget / int(row_bytes);
      if (stages > kMaxStages) stages = kMaxStages;
      if (stages < 2) stages = 2;
      const int smem = kBarrierBytes + stages * int(row_bytes);
      int grid = device_info().sm_count * bf16_ctas_per_sm(smem);
      if (grid > a.T) grid = a.T;
      st = launch_pdl(dispatch_bf16_kernel, dim3(grid), dim3(32), smem, stream,
                      static_cast<const uint8_t*>(a.x), a.topk_weights, a.slot_of,
                      a.T, a.K, row_bytes, stages, static_cast<uint8_t*>(a.recv_x),
                      a.recv_w, a.err);
    } else {
      const int nvec = a.H / 8;
      int threads = nvec < 1024 ? ((nvec + 31) / 32) * 32 : 1024;
      st = launch_pdl(dispatch_fp8_kernel, dim3(a.T), dim3(threads), 0, stream,
                      static_cast<const uint4*>(a.x), a.topk_weights, a.slot_of,
                      a.T, a.H, a.K, static_cast<uint8_t*>(a.recv_x), a.recv_scale,
                      a.recv_w);
    }
    if (st != cudaSuccess) return st;
  }
  if (a.zero_padding) {
    const int64_t row_bytes = a.fp8 ? int64_t(a.H) : int64_t(a.H) * 2;
    int grid = a.E < 1024 ? a.E : 1024;
    st = launch_pdl(zero_padding_kernel, dim3(grid), dim3(256), 0, stream,
                    a.expert_start, a.expert_end, a.E, row_bytes,
                    a.fp8 ? a.H / 128 : 0, static_cast<uint8_t*>(a.recv_x),
                    a.fp8 ? a.recv_scale : nullptr, a.recv_w);
    if (st != cudaSuccess) return st;
  }
  return cudaSuccess;
}

}  // namespace ep

// Device-side helpers shared by the sm_103a kernels: bulk-copy (TMA) and
// mbarrier wrappers in inline PTX, bounded waits, the device error word.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ep {

// Bits of the device error word (layout->err).  The host maps them to
// ep_status codes, most severe routing error first.
enum : int32_t {
  ERRBIT_EXPERT_RANGE = 1,
  ERRBIT_DUP_EXPERT = 2,
  ERRBIT_TIMEOUT = 4,
  // a wait gave up and the bulk copies its CTA had issued were still not
  // complete when it returned (they may land in shared memory after it)
  ERRBIT_TIMEOUT_PENDING = 8,
};

// Default limit of one on-chip wait.  Far above any legitimate latency; a
// wait that runs out records ERRBIT_TIMEOUT and the kernel returns.
constexpr uint64_t kWaitTimeoutNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// ---- programmatic dependent launch ----------------------------------------
// Every kernel of the library is launched with programmatic stream
// serialisation and waits for the preceding grid (griddepcontrol.wait)
// before its first read of global memory that another kernel may have
// written.  None signals its dependents early: the next grid starts
// launching as this one's CTAs exit, which still hides the launch gap.  An
// early signal let waiting CTAs of the next grid hold warp slots while this
// grid ran (measured, same box: prefill step 178 -> 174 us, skew
// 134 -> 128 us, 16K-token FP8 step 544 -> 518 us without it).

__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---- mbarrier -----------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(count)
               : "memory");
}

// Makes initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of `bar` to complete.  Bounded twice: by the
// global timer (timeout_ns) and, should the timer not advance, by an
// iteration count.  Returns false if the wait gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t outer = 0; outer < (1u << 22); ++outer) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > timeout_ns) return false;
  }
  return false;
}

// ---- bulk copies (non-tensor TMA) --------------------------------------
// Both addresses 16-byte aligned, size a multiple of 16 bytes.

// global -> shared, completion counted on `bar` (complete_tx bytes).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src,
                                          uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// ---- per-thread asynchronous copies ---------------------------------------
// 16 bytes global -> shared (both 16-byte aligned), cached in L2 only; the
// issuing thread's copies are complete after cp_async_wait_all, and visible
// to the CTA after a barrier that follows it.  Completion is tracked by the
// hardware like a load's, so there is no flag to wait on.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---- streaming global access ---------------------------------------------

// Row-split kernels: a token's row of 16-byte vectors is shared by
// gridDim.y CTAs; the CTA's threads start at first_vec() and step by
// vec_stride().
__device__ __forceinline__ int first_vec() { return blockIdx.y * blockDim.x + threadIdx.x; }
__device__ __forceinline__ int vec_stride() { return blockDim.x * gridDim.y; }

// 16-byte read-only load that does not allocate in L1 (data read once).
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Two adjacent 16-byte vectors in one 256-bit load (p 32-byte aligned): a
// warp's request then covers each 32-byte sector once, which matters where
// a sector read twice crosses the link twice (rows in host memory).
__device__ __forceinline__ void ld_stream_u4x2(const void* p, uint4& a, uint4& b) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z),
                 "=r"(b.w)
               : "l"(p));
}

// ---- numerics ------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) {
  return __uint_as_float(w << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t w) {
  return __uint_as_float(w & 0xFFFF0000u);
}

// Two fp32 -> packed bf16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two fp32 -> packed E4M3x2 (round to nearest even, saturate to +-448);
// `lo` in the low byte.
__device__ __forceinline__ uint16_t pack_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void record_error(int32_t* err, int32_t bit) {
  if (err) atomicOr(err, bit);
}

}  // namespace ep

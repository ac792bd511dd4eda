// E4M3 quantisation of bf16 rows in 1x128 blocks ("Deep Dive - DeepEP",
// "Precision: FP8 on the wire, BF16 for the reduction": one fp32 scale per
// 128 values), shared by the dispatch kernels.
#pragma once

#include "ep_device.cuh"

namespace ep {

// x / s for a block scale s in [kFastScaleMin, FLT_MAX] and |x| <= 448 s,
// given y = RN(1/s): q0 = x * y, then one correction with the exact residual
// r = x - q0 * s (one FMA), after Markstein's FMA-based division
// (P. Markstein, "IA-64 and Elementary Functions", 2000).  The reciprocal
// is taken once per block.  The quotient can differ from the IEEE one in
// the last fp32 bit, but never in the E4M3 code it rounds to: the inputs
// here are bf16 values and the scale of a bf16 block maximum, and
// ep_selftest_fp8_quotient compares the codes against those of the IEEE
// division over that whole domain (every bf16 maximum, every bf16 value).
constexpr float kFastScaleMin = 0x1p-100f;

__device__ __forceinline__ float scaled_quotient(float x, float s, float y) {
  const float q0 = x * y;
  const float r = fmaf(-q0, s, x);
  // s > 0: the quotient has x's sign (the correction would turn -0 into +0)
  return copysignf(fmaf(r, y, q0), x);
}

// The quotient x / s of one block, by the fast form where it holds and by
// IEEE division elsewhere: below kFastScaleMin 1/s would overflow, and an
// infinite scale (a block holding +-inf) would make the residual inf - inf;
// there the division gives +-0 for finite x and NaN for +-inf, as the
// definition does.
struct BlockQuotient {
  float s, y;
  bool fast;
  __device__ __forceinline__ explicit BlockQuotient(float scale)
      : s(scale), y(0.0f), fast(scale >= kFastScaleMin && scale <= 0x1.fffffep127f) {
    if (fast) y = __frcp_rn(scale);
  }
  __device__ __forceinline__ float operator()(float x) const {
    return fast ? scaled_quotient(x, s, y) : __fdiv_rn(x, s);
  }
};

// One 16-channel group of a row (two 16-byte bf16 vectors r0, r1; zeros for
// a lane past the row): 8 aligned lanes hold one 128-channel block.  The
// block's exact amax comes from three shuffles, scale = amax / 448 (fp32,
// round to nearest; 0 for an all-zero block), and the 16 E4M3 codes of
// x / scale (round to nearest even, saturating) are packed into *q.  All 32
// lanes of the warp call.
__device__ __forceinline__ void quantize_group16(uint4 r0, uint4 r1, uint4* q, float* scale) {
  const float f[16] = {bf16_lo(r0.x), bf16_hi(r0.x), bf16_lo(r0.y), bf16_hi(r0.y),
                       bf16_lo(r0.z), bf16_hi(r0.z), bf16_lo(r0.w), bf16_hi(r0.w),
                       bf16_lo(r1.x), bf16_hi(r1.x), bf16_lo(r1.y), bf16_hi(r1.y),
                       bf16_lo(r1.z), bf16_hi(r1.z), bf16_lo(r1.w), bf16_hi(r1.w)};
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(f[j]));
#pragma unroll
  for (int o = 4; o >= 1; o >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  *q = make_uint4(0, 0, 0, 0);
  *scale = 0.0f;
  if (amax != 0.0f) {
    const float s = __fdiv_rn(amax, 448.0f);
    const BlockQuotient div(s);
    uint32_t p[8];
    if (div.fast) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        p[j] = pack_e4m3x2(scaled_quotient(f[2 * j], s, div.y),
                           scaled_quotient(f[2 * j + 1], s, div.y));
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        p[j] = pack_e4m3x2(__fdiv_rn(f[2 * j], s), __fdiv_rn(f[2 * j + 1], s));
    }
    *q = make_uint4(p[0] | (p[1] << 16), p[2] | (p[3] << 16), p[4] | (p[5] << 16),
                    p[6] | (p[7] << 16));
    *scale = s;
  }
}

}  // namespace ep

// f8_convert.cuh -- the 1x128 / 128x128 quantisers' per-element arithmetic,
// shared by the quantiser kernels and by the decode GEMM that quantises its
// activations on load: x / s as an IEEE FP32 division (round to nearest),
// then the hardware's round-to-nearest-even, saturating FP8 conversion
// ("news.rkmt.cn/news/5092" section 5.2: s = amax / 448 per block;
// "lpnh.cn/news/2822121" section 6.3: round to nearest).
#pragma once

#include <cstdint>

#include "common.cuh"

namespace fp8gemm {

// Two FP32 values -> two FP8 bytes (lo in the low byte), round to nearest
// even, saturate to the format's largest finite value (+-448 e4m3, +-57344
// e5m2).
template <bool kE5M2>
__device__ __forceinline__ uint32_t cvt_f8x2(float lo, float hi) {
  uint16_t r;
  if constexpr (kE5M2)
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// The format's largest finite value: the divisor of the scale rule.
template <bool kE5M2>
__device__ __forceinline__ float f8_limit() {
  return kE5M2 ? 57344.0f : kE4M3Max;
}

// Four values -> four FP8 bytes (x / s each); kCount: adds to n the
// quotients the conversion clamps (not within +-limit, NaN included).
template <bool kE5M2, bool kCount = false>
__device__ __forceinline__ uint32_t quant4(float4 v, float s, unsigned* n = nullptr) {
  const float q0 = __fdiv_rn(v.x, s), q1 = __fdiv_rn(v.y, s);
  const float q2 = __fdiv_rn(v.z, s), q3 = __fdiv_rn(v.w, s);
  if constexpr (kCount) {
    const float lim = f8_limit<kE5M2>();
    *n += unsigned(!(fabsf(q0) <= lim)) + unsigned(!(fabsf(q1) <= lim)) +
          unsigned(!(fabsf(q2) <= lim)) + unsigned(!(fabsf(q3) <= lim));
  }
  return cvt_f8x2<kE5M2>(q0, q1) | (cvt_f8x2<kE5M2>(q2, q3) << 16);
}

// quant4 through the block's reciprocal r = RN(1 / s): q' = RN(x * r) is
// within 2.5 units in the last place of RN(x / s) (two roundings of relative
// size 2^-24 each, plus the half unit of RN(x / s) itself), and every point
// where the FP8 conversion changes its result -- the values and midpoints of
// e4m3 and e5m2, normal and subnormal, and the limits 448 and 57344 -- has its
// low 19 fraction bits zero.  So a finite q' whose low 19 fraction bits are at
// least 8 away from zero (mod 2^19), or an exact zero, converts and counts
// exactly as RN(x / s) does; when any of the four is not, all four are divided.
template <bool kE5M2, bool kCount = false>
__device__ __forceinline__ uint32_t quant4_recip(float4 v, float s, float r,
                                                 unsigned* n = nullptr) {
  const float q0 = __fmul_rn(v.x, r), q1 = __fmul_rn(v.y, r);
  const float q2 = __fmul_rn(v.z, r), q3 = __fmul_rn(v.w, r);
  auto sure = [](float q) {
    const uint32_t b = __float_as_uint(q);
    const uint32_t f = b & 0x7FFFFu;
    return (b & 0x7F800000u) != 0x7F800000u && ((b & 0x7FFFFFFFu) == 0 || f - 8u <= 0x7FFF0u);
  };
  if (!(sure(q0) && sure(q1) && sure(q2) && sure(q3))) return quant4<kE5M2, kCount>(v, s, n);
  if constexpr (kCount) {
    const float lim = f8_limit<kE5M2>();
    *n += unsigned(fabsf(q0) > lim) + unsigned(fabsf(q1) > lim) + unsigned(fabsf(q2) > lim) +
          unsigned(fabsf(q3) > lim);
  }
  return cvt_f8x2<kE5M2>(q0, q1) | (cvt_f8x2<kE5M2>(q2, q3) << 16);
}

__device__ __forceinline__ float absmax4(float4 v) {
  return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

}  // namespace fp8gemm

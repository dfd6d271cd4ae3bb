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

__device__ __forceinline__ float absmax4(float4 v) {
  return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

}  // namespace fp8gemm

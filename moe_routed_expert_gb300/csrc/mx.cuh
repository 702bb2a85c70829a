// MX (microscaling) quantisation of 32-element groups, as "MegaMoE",
// "A8W8-FP 量化场景" and "A4W4-FP 量化场景" use it: a shared E8M0 exponent per
// group and FP8 (E4M3FN or E5M2) or FP4 (E2M1) elements.
//
// Shared exponent: X = 2^(floor(log2 amax) - emax), emax = 8 (E4M3), 15
// (E5M2) or 2 (E2M1), clamped below at 2^-127; a group holding an infinity or
// a NaN gets the NaN scale 0xFF.  Elements: x / X rounded to nearest even with
// saturation to the largest finite value (the hardware's satfinite convert;
// E2M1 has no NaN, and a NaN converts to the largest positive code, 7).
// floor(log2 amax) is read off amax's exponent field, so the decision is exact.
#pragma once

#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "moe_mx.h"

namespace moe {

template <int FMT>
struct Fp8Fmt;
template <>
struct Fp8Fmt<MOE_FP8_E4M3> {
  static constexpr int emax = 8;
  static constexpr __nv_fp8_interpretation_t kind = __NV_E4M3;
};
template <>
struct Fp8Fmt<MOE_FP8_E5M2> {
  static constexpr int emax = 15;
  static constexpr __nv_fp8_interpretation_t kind = __NV_E5M2;
};

template <>
struct Fp8Fmt<MOE_FP4_E2M1> {
  static constexpr int emax = 2;
};

// E8M0 code of a group whose largest magnitude has bit pattern `amax_bits`
// (sign cleared; any infinity or NaN compares above every finite value), and
// the multiplier 2^-e that maps the group onto the element grid.
template <int FMT>
__device__ __forceinline__ uint32_t mx_scale_code(uint32_t amax_bits, float& inv) {
  const int ef = static_cast<int>(amax_bits >> 23);
  if (ef == 0xFF) {
    inv = __uint_as_float(0x7FC00000u);
    return 0xFFu;
  }
  int e = ef - 127 - Fp8Fmt<FMT>::emax;  // a zero or subnormal amax lands below -127
  if (e < -127) e = -127;
  inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, a normal float for e in [-127, 119]
  return static_cast<uint32_t>(e + 127);
}

// Two floats -> two fp8 codes, the first in the low byte.
template <int FMT>
__device__ __forceinline__ uint32_t fp8x2(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, Fp8Fmt<FMT>::kind));
}

// Quantise 32 values: codes into q (element i in byte i % 4 of word i / 4),
// returns the scale code.
template <int FMT>
__device__ __forceinline__ uint32_t mx_quant32(const float (&v)[32], uint32_t (&q)[8]) {
  uint32_t amax = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = max(amax, __float_as_uint(v[i]) & 0x7FFFFFFFu);
  float inv;
  const uint32_t sc = mx_scale_code<FMT>(amax, inv);
#pragma unroll
  for (int w = 0; w < 8; ++w)
    q[w] = fp8x2<FMT>(v[4 * w] * inv, v[4 * w + 1] * inv) | (fp8x2<FMT>(v[4 * w + 2] * inv, v[4 * w + 3] * inv) << 16);
  return sc;
}

// Quantise 32 values to E2M1: element i in nibble i % 8 of word i / 8 (two
// elements per byte, the first in the low nibble); returns the scale code.
__device__ __forceinline__ uint32_t mx_quant32_fp4(const float (&v)[32], uint32_t (&q)[4]) {
  uint32_t amax = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = max(amax, __float_as_uint(v[i]) & 0x7FFFFFFFu);
  float inv;
  const uint32_t sc = mx_scale_code<MOE_FP4_E2M1>(amax, inv);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float2 pr = make_float2(v[8 * w + 2 * b] * inv, v[8 * w + 2 * b + 1] * inv);
      word |= static_cast<uint32_t>(__nv_cvt_float2_to_fp4x2(pr, __NV_E2M1, cudaRoundNearest)) << (8 * b);
    }
    q[w] = word;
  }
  return sc;
}

}  // namespace moe

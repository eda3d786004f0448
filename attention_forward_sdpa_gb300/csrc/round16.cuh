// round16.cuh -- the epilogue's fp32 -> 16-bit output rounding, in the three
// modes of "MoonMath.ai abre un nucleo de atencion HIP para AMD MI300X ..."
// (7minutos.es), section "Punto de referencia": RTNE (nearest, ties to even),
// RTNA (nearest, ties away from zero) and RTZ (toward zero).  Overflow follows
// IEEE 754; NaN stays NaN.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace attn {

enum RoundMode : int { kRTNE = 0, kRTNA = 1, kRTZ = 2 };

__device__ __forceinline__ uint16_t round_bf16(float x, int mode) {
  if (mode == kRTZ) return __bfloat16_as_ushort(__float2bfloat16_rz(x));
  if (mode == kRTNA) {
    const uint32_t u = __float_as_uint(x);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);  // NaN
    // bf16 keeps binary32's exponent field, so adding half of the dropped
    // unit to the pattern and truncating rounds the magnitude half-up; a carry
    // out of the fraction moves to the next binade (or to infinity) as it must.
    return (uint16_t)((u + 0x8000u) >> 16);
  }
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint16_t round_f16(float x, int mode) {
  if (mode == kRTZ) return __half_as_ushort(__float2half_rz(x));
  const uint16_t rn = __half_as_ushort(__float2half_rn(x));
  if (mode != kRTNA) return rn;
  const uint16_t rz = __half_as_ushort(__float2half_rz(x));
  if (rn != rz) return rn;  // nearest already lies away from zero: same for RTNA
  // rn == rz: either |x| is below the midpoint (RTNA agrees) or |x| is exactly
  // the midpoint and the even neighbour lies toward zero (RTNA goes away).
  if ((rz & 0x7C00u) == 0x7C00u) return rz;  // inf / NaN
  const float ax = fabsf(x);
  const float lo = fabsf(__half2float(__ushort_as_half(rz)));
  const uint16_t away_bits = (uint16_t)(rz + 1u);  // next magnitude, same sign
  if ((away_bits & 0x7FFFu) == 0x7C00u) {          // away neighbour is infinity
    return ax == 65520.0f ? away_bits : rz;
  }
  const float hi = fabsf(__half2float(__ushort_as_half(away_bits)));
  // lo <= ax < hi lie within one binade step, so both differences are exact.
  return (ax - lo == hi - ax) ? away_bits : rz;
}

template <bool BF16>
__device__ __forceinline__ uint16_t round_out(float x, int mode) {
  if constexpr (BF16) return round_bf16(x, mode);
  else return round_f16(x, mode);
}

template <bool BF16>
__device__ __forceinline__ uint32_t round_out_x2(float lo, float hi, int mode) {
  return (uint32_t)round_out<BF16>(lo, mode) | ((uint32_t)round_out<BF16>(hi, mode) << 16);
}

}  // namespace attn

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

// 32 fp32 accumulator columns times scale -> 16 packed 16-bit pairs (even
// column in the low half), with the mode tested once for the whole row chunk.
// RTNE and RTZ use the packed conversions; bf16 RTNA adds half of the dropped
// unit to the binary32 pattern (NaN kept quiet), fp16 RTNA takes the scalar
// path above.
template <bool BF16>
__device__ __forceinline__ uint32_t cvt_pack_rn(float lo, float hi) {
  uint32_t r;
  if constexpr (BF16) asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  else asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <bool BF16>
__device__ __forceinline__ uint32_t cvt_pack_rz(float lo, float hi) {
  uint32_t r;
  if constexpr (BF16) asm("cvt.rz.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  else asm("cvt.rz.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t bf16_rna_bits(float x) {
  const uint32_t u = __float_as_uint(x);
  const uint32_t nan = (u >> 16) | 0x0040u;
  const uint32_t rounded = (u + 0x8000u) >> 16;
  return (u & 0x7FFFFFFFu) > 0x7F800000u ? nan : rounded;
}

template <bool BF16>
__device__ __forceinline__ void round_pack32(const uint32_t (&o)[32], float scale, int mode,
                                             uint32_t (&w)[16]) {
  if (mode == kRTNE) {
#pragma unroll
    for (int e = 0; e < 16; ++e)
      w[e] = cvt_pack_rn<BF16>(__uint_as_float(o[2 * e]) * scale, __uint_as_float(o[2 * e + 1]) * scale);
  } else if (mode == kRTZ) {
#pragma unroll
    for (int e = 0; e < 16; ++e)
      w[e] = cvt_pack_rz<BF16>(__uint_as_float(o[2 * e]) * scale, __uint_as_float(o[2 * e + 1]) * scale);
  } else if constexpr (BF16) {
#pragma unroll
    for (int e = 0; e < 16; ++e)
      w[e] = bf16_rna_bits(__uint_as_float(o[2 * e]) * scale) |
             (bf16_rna_bits(__uint_as_float(o[2 * e + 1]) * scale) << 16);
  } else {
#pragma unroll
    for (int e = 0; e < 16; ++e)
      w[e] = round_out_x2<false>(__uint_as_float(o[2 * e]) * scale, __uint_as_float(o[2 * e + 1]) * scale,
                                 kRTNA);
  }
}

}  // namespace attn

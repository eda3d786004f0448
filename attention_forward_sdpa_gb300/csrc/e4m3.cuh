// e4m3.cuh -- widening of fp8 E4M3 codes (1 sign, 4 exponent bits with bias
// 7, 3 fraction bits, S.1111.111 = NaN, no infinities) to the 16-bit formats
// the MMAs read.  Every E4M3 value is exact in fp16 and in bf16, so the
// conversion unit's e4m3x2 -> f16x2 step is exact, and so is the route on to
// bf16 through f32.  NaN codes give NaN, as the format defines them.
//
// (A placement of the code's bits into the target's exponent and fraction
// fields followed by one power-of-two multiply costs fewer instructions but
// turns the NaN codes into +-480; making it NaN-correct doubled its integer
// work, and a 16-code test that skipped the fix-up for blocks without NaN
// codes slowed the fp8 decode further, so the conversion unit does the work.)
#pragma once

#include <cstdint>

namespace attn {

// Two codes (the low 16 bits of w, low byte first) -> f16x2 on the
// conversion unit.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w) {
  uint32_t r;
  const uint16_t c = (uint16_t)w;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(c));
  return r;
}

// Two codes (the low 16 bits of w) -> bf16x2 through the conversion unit:
// f16x2 (exact), each half to f32 (exact), both to bf16 (exact: three
// fraction bits fit).  NaN codes give NaN at the first step and stay NaN.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t w) {
  const uint32_t h = e4m3x2_to_f16x2(w);
  float lo, hi;
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h));
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 16 codes -> 16 values in element order (lo: codes 0-7, hi: codes 8-15),
// on the conversion unit (NaN codes give NaN).
template <bool BF16>
__device__ __forceinline__ void e4m3x16_widen(const uint4 w, uint4& lo, uint4& hi) {
  if constexpr (BF16) {
    lo.x = e4m3x2_to_bf16x2(w.x);
    lo.y = e4m3x2_to_bf16x2(w.x >> 16);
    lo.z = e4m3x2_to_bf16x2(w.y);
    lo.w = e4m3x2_to_bf16x2(w.y >> 16);
    hi.x = e4m3x2_to_bf16x2(w.z);
    hi.y = e4m3x2_to_bf16x2(w.z >> 16);
    hi.z = e4m3x2_to_bf16x2(w.w);
    hi.w = e4m3x2_to_bf16x2(w.w >> 16);
  } else {
    lo.x = e4m3x2_to_f16x2(w.x);
    lo.y = e4m3x2_to_f16x2(w.x >> 16);
    lo.z = e4m3x2_to_f16x2(w.y);
    lo.w = e4m3x2_to_f16x2(w.y >> 16);
    hi.x = e4m3x2_to_f16x2(w.z);
    hi.y = e4m3x2_to_f16x2(w.z >> 16);
    hi.z = e4m3x2_to_f16x2(w.w);
    hi.w = e4m3x2_to_f16x2(w.w >> 16);
  }
}

}  // namespace attn

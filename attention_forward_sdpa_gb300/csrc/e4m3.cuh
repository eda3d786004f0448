// e4m3.cuh -- widening of fp8 E4M3 codes (1 sign, 4 exponent bits with bias
// 7, 3 fraction bits) to the 16-bit formats the MMAs read, by bit placement
// on the integer and FMA pipes rather than the conversion unit.
//
// A code s.eeee.mmm read as the low byte of a 16-bit lane, sign-extended to
// the whole lane and shifted so that eeee.mmm lands where the target format
// keeps its low exponent bits and top fraction bits, is a value of that
// format equal to the code's value times a fixed power of two: 2^-8 for fp16
// (exponent bias 15 - 7) and 2^-120 for bf16 (127 - 7).  This holds for
// normal codes and for the subnormal ones (e = 0), which land on subnormals
// of the target with the same fraction.  One multiply by 2^8 or 2^120 in the
// target format then gives the value exactly (no rounding: a power of two,
// no overflow; subnormal inputs are honoured by mul.rn without .ftz).
//
// The two NaN codes (S.1111.111) would land on +-480 that way (no finite
// code is 480: the largest is 448), so before the multiply the lanes whose
// placed bits are all ones get the rest of the target's exponent field set,
// which makes them NaN (and the product NaN).  Detection without a compare:
// adding one unit of the lowest placed bit to the masked field carries out
// of it only when every placed bit is one.
#pragma once

#include <cstdint>

namespace attn {

// Codes b_lo, b_hi (bytes `sel` picks from w) -> two 16-bit values, low half
// from b_lo.  sel is a prmt selector whose bytes are (b_lo, sign(b_lo),
// b_hi, sign(b_hi)).
template <bool BF16>
__device__ __forceinline__ uint32_t e4m3x2_widen(uint32_t w, uint32_t sel) {
  uint32_t x, r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(x) : "r"(w), "r"(sel));
  if constexpr (BF16) {
    uint32_t y = (x << 4) & 0x87F087F0u;          // s | eeee.mmm at bits 10..4: value * 2^-120
    // NaN codes: bits 10..4 all set -> the carry lands in bit 11; 15 * 0x0800
    // sets bits 14..11, completing the all-ones exponent (no lane overflows)
    const uint32_t nan = ((y & 0x07F007F0u) + 0x00100010u) & 0x08000800u;
    y += nan * 15u;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(y), "r"(0x7B807B80u));   // * 2^120
  } else {
    uint32_t y = (x << 7) & 0xBF80BF80u;          // s | eeee.mmm at bits 13..7: value * 2^-8
    // NaN codes: bits 13..7 all set -> the carry is bit 14, the one exponent
    // bit still clear
    const uint32_t nan = ((y & 0x3F803F80u) + 0x00800080u) & 0x40004000u;
    y += nan;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(y), "r"(0x5C005C00u));    // * 2^8
  }
  return r;
}

// Selectors: codes (0, 1) and (2, 3) of a 32-bit word, each followed by its
// replicated sign byte (prmt selector nibbles with the top bit set).
constexpr uint32_t kSelLo = 0x9180u;
constexpr uint32_t kSelHi = 0xB3A2u;

// 16 codes -> 16 values in element order (lo: codes 0-7, hi: codes 8-15)
template <bool BF16>
__device__ __forceinline__ void e4m3x16_widen(const uint4 w, uint4& lo, uint4& hi) {
  lo.x = e4m3x2_widen<BF16>(w.x, kSelLo);
  lo.y = e4m3x2_widen<BF16>(w.x, kSelHi);
  lo.z = e4m3x2_widen<BF16>(w.y, kSelLo);
  lo.w = e4m3x2_widen<BF16>(w.y, kSelHi);
  hi.x = e4m3x2_widen<BF16>(w.z, kSelLo);
  hi.y = e4m3x2_widen<BF16>(w.z, kSelHi);
  hi.z = e4m3x2_widen<BF16>(w.w, kSelLo);
  hi.w = e4m3x2_widen<BF16>(w.w, kSelHi);
}

}  // namespace attn

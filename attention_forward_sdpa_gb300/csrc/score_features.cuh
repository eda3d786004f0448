// score_features.cuh -- the feature-flagged score rewrites and the sink term
// shared by the prefill kernels and both decode kernels ("gfx942 unified
// attention, from the math up", sec. 9 names softcap, ALiBi and sinks; the
// definitions are the usual ones, stated in include/attn_fwd.h).
#pragma once

#include <cstdint>

#include "sm103_ptx.cuh"

namespace attn {

// One scaled score x = tau * q.k: softcap, then the ALiBi bias -slope * dist.
// The cap uses the MUFU tanh: its relative error (about 2^-11) moves a capped
// score y by at most |y| * 2^-11 (< cap * 2^-11), so each probability moves by
// that relative amount, a fifth of the 2^-9 relative step of a bf16 output.
__device__ __forceinline__ float rewrite_score(float x, float cap, float inv_cap, float slope,
                                               float dist) {
  if (cap > 0.f) x = cap * fast_tanh(x * inv_cap);
  return fmaf(-slope, fabsf(dist), x);
}

// A row of raw scores q.k (fp32 bit patterns in s[c][e], key column 32c + e
// of the NC * 32 columns passed): each becomes (rewrite(tau * q.k)) / tau, so that the softmax that
// follows, which multiplies by tau * log2(e), sees the rewritten score.  d0 is
// the distance from the row's aligned key to column 0 (diag - first key).
// The constants are folded so that an element costs one multiply, one MUFU
// tanh and one FMA: (cap / tau) * tanh(q.k * tau / cap) - (slope / tau) * |dist|.
template <int NC>
__device__ __forceinline__ void rewrite_scores(uint32_t (&s)[NC][32], float tau, float cap,
                                               float slope, float d0) {
  const float inv_tau = 1.f / tau;
  const float ks = -slope * inv_tau;
  if (cap > 0.f) {
    const float a = tau / cap;
    const float b = cap * inv_tau;
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float t = fast_tanh(__uint_as_float(s[c][e]) * a);
        s[c][e] = __float_as_uint(fmaf(ks, fabsf(d0 - (float)(32 * c + e)), t * b));
      }
  } else {
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
      for (int e = 0; e < 32; ++e)
        s[c][e] = __float_as_uint(fmaf(ks, fabsf(d0 - (float)(32 * c + e)), __uint_as_float(s[c][e])));
  }
}

// Final normalisation of a row: m is the running reference max (log2 units),
// l the running denominator, sink the row's sink logit (natural units, -inf
// for none).  Gives the factor that turns o into O and the natural-log
// log-sum-exp: O = o / (l + 2^(z log2 e - m)), both formed against
// M = max(m, z log2 e) so that nothing overflows.  A row with no visible key
// (m = -inf) gets O = 0 and lse = z (-inf without a sink).
__device__ __forceinline__ void finish_row(float m, float l, float sink, float& inv_l, float& lse) {
  constexpr float kLn2f = 0.693147180559945309f;
  constexpr float kLog2ef = 1.4426950408889634f;
  if (sink == -INFINITY) {
    // l == 0: no visible key; a NaN l (from a NaN score) gives NaN, as the
    // definition does
    inv_l = l != 0.f ? 1.f / l : 0.f;
    lse = l != 0.f ? m * kLn2f + logf(l) : -INFINITY;
    return;
  }
  const float zl = sink * kLog2ef;
  const float M = fmaxf(m, zl);
  const float a = m == -INFINITY ? 0.f : exp2f(m - M);
  const float lt = fmaf(l, a, exp2f(zl - M));
  inv_l = a / lt;
  lse = (M + log2f(lt)) * kLn2f;
}

}  // namespace attn

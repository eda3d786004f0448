// score_features.cuh -- the feature-flagged score rewrites and the sink term
// shared by the prefill kernels and the SIMT decode kernel ("gfx942 unified
// attention, from the math up", sec. 9 names softcap, ALiBi and sinks; the
// definitions are the usual ones, stated in include/attn_fwd.h).
#pragma once

#include <cstdint>

#include "sm103_ptx.cuh"

namespace attn {

// tanh(y) = 1 - 2 / (e^(2y) + 1), from the exponential (an identity, not a
// library routine).  |y| is clamped to 10, where tanh is +-1 to within fp32
// rounding, so that e^(2y) stays finite.  Absolute error ~1e-7, which is
// what matters for a capped logit.
__device__ __forceinline__ float tanh_via_exp2(float y) {
  const float yc = fminf(fmaxf(y, -10.f), 10.f);
  const float e = fast_exp2(yc * 2.8853900817779268f);   // 2 * log2(e)
  return 1.f - __fdividef(2.f, e + 1.f);
}

// One scaled score x = tau * q.k: softcap, then the ALiBi bias -slope * dist.
__device__ __forceinline__ float rewrite_score(float x, float cap, float inv_cap, float slope,
                                               float dist) {
  if (cap > 0.f) x = cap * tanh_via_exp2(x * inv_cap);
  return fmaf(-slope, fabsf(dist), x);
}

// A tile row of raw scores q.k (fp32 bit patterns in s[c][e], key column
// 32c + e): each becomes (rewrite(tau * q.k)) / tau, so that the softmax that
// follows, which multiplies by tau * log2(e), sees the rewritten score.  d0 is
// the distance from the row's aligned key to column 0 (diag - first key).
__device__ __forceinline__ void rewrite_scores(uint32_t (&s)[4][32], float tau, float cap,
                                               float slope, float d0) {
  const float inv_tau = 1.f / tau;
  const float inv_cap = cap > 0.f ? 1.f / cap : 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float x = __uint_as_float(s[c][e]) * tau;
      s[c][e] = __float_as_uint(rewrite_score(x, cap, inv_cap, slope, d0 - (float)(32 * c + e)) * inv_tau);
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
    inv_l = l > 0.f ? 1.f / l : 0.f;
    lse = l > 0.f ? m * kLn2f + logf(l) : -INFINITY;
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

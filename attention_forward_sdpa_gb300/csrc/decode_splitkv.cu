// decode_splitkv.cu -- split-KV decode ("gfx942 unified attention, from the
// math up", sec. 8): one query row per (sequence, q head); the key range of a
// sequence is cut into num_splits contiguous parts handled by separate CTAs,
// each producing a partial online-softmax state (un-normalised o, running max
// m, denominator l); a second kernel merges the parts by the log-sum-exp rule
// and rounds the result.
//
// Decode is a bandwidth problem: every K/V byte is read once and used for
// 2 * GH flops (GH = query heads sharing the KV head), so the kernel is built
// around coalesced row loads: lane i of a warp owns channels
// [i*D/32, (i+1)*D/32) of every K and V row; a warp walks chunks of CK keys
// (a chunk never crosses a page because block sizes are multiples of 16); the
// per-key dot products of a chunk are reduced across the warp by a
// transposing butterfly (each step halves the vector, so the shuffle count is
// about one per dot product), and the softmax bookkeeping of the chunk runs on
// GH lanes from shared memory.  The warps of a CTA keep separate states that
// are merged in a fixed order at the end.
//
// This SIMT kernel serves the shapes the tcgen05 decode (decode_tcgen05.cu)
// does not take: group sizes that are neither a power of two up to 16 nor a
// multiple of 16, and fp8 caches at head sizes 64 and 256.  The file also holds the merge kernel that
// both split kernels use (one warp per (sequence, head): every split's (m, l)
// in one round trip, up to eight partial rows in flight, splits merged in a
// fixed order) and the elementwise rounding kernel behind attn_round_f32.

#include <algorithm>
#include <type_traits>

#include "attn_internal.h"
#include "round16.cuh"
#include "score_features.cuh"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kDecWarps = 8;
constexpr float kLn2 = 0.693147180559945309f;

// One level of the butterfly reduce-scatter of N per-lane partial sums: the
// vector of CUR live entries is halved, each lane keeping the half selected
// by its MASK bit and adding the partner's copy of it.  When one entry is
// left the remaining levels are plain butterflies.  Afterwards lane L holds
// the complete sum of entry L*(N/32)+k in v[k] for N >= 32, or of entry
// L / (32/N) in v[0] for N < 32.
template <int N, int CUR, int MASK>
__device__ __forceinline__ void scatter_step(float (&v)[N], int lane) {
  if constexpr (MASK >= 1) {
    if constexpr (CUR > 1) {
      constexpr int kHalf = CUR / 2;
      const bool upper = (lane & MASK) != 0;
#pragma unroll
      for (int i = 0; i < kHalf; ++i) {
        const float send = upper ? v[i] : v[i + kHalf];
        const float keep = upper ? v[i + kHalf] : v[i];
        v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, MASK);
      }
      scatter_step<N, kHalf, MASK / 2>(v, lane);
    } else {
      v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], MASK);
      scatter_step<N, 1, MASK / 2>(v, lane);
    }
  }
}

template <int N>
__device__ __forceinline__ int scatter_index(int lane, int k) {
  if constexpr (N >= 32) return lane * (N / 32) + k;
  else return lane / (32 / N);
}

template <bool BF16>
__device__ __forceinline__ void widen2(uint32_t w, float& lo, float& hi) {
  if constexpr (BF16) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
  } else {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w));
    lo = a.x;
    hi = a.y;
  }
}

template <bool BF16, int DPL>
__device__ __forceinline__ void load_row(const uint16_t* __restrict__ src, float (&x)[DPL]) {
  if constexpr (DPL == 8) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(src));
    widen2<BF16>(w.x, x[0], x[1]);
    widen2<BF16>(w.y, x[2], x[3]);
    widen2<BF16>(w.z, x[4], x[5]);
    widen2<BF16>(w.w, x[6], x[7]);
  } else if constexpr (DPL == 4) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
    if constexpr (BF16) {
      x[0] = __uint_as_float(w.x << 16);
      x[1] = __uint_as_float(w.x & 0xFFFF0000u);
      x[2] = __uint_as_float(w.y << 16);
      x[3] = __uint_as_float(w.y & 0xFFFF0000u);
    } else {
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
      const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
      x[0] = a.x; x[1] = a.y; x[2] = c.x; x[3] = c.y;
    }
  } else {
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(src));
    if constexpr (BF16) {
      x[0] = __uint_as_float(w << 16);
      x[1] = __uint_as_float(w & 0xFFFF0000u);
    } else {
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w));
      x[0] = a.x; x[1] = a.y;
    }
  }
}

// Two E4M3 codes (low byte first) -> two floats.  The conversion to f16x2 is
// exact (every E4M3 value is an fp16 normal or zero), and so is the widening.
__device__ __forceinline__ void widen_e4m3x2(uint32_t two_codes, float& lo, float& hi) {
  uint32_t h;
  const uint16_t c = (uint16_t)two_codes;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(c));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h));
  lo = a.x;
  hi = a.y;
}

// DPL fp8 codes of a lane's channels -> floats (fp8 caches)
template <int DPL>
__device__ __forceinline__ void load_row8(const uint8_t* __restrict__ src, float (&x)[DPL]) {
  if constexpr (DPL == 8) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
    widen_e4m3x2(w.x, x[0], x[1]);
    widen_e4m3x2(w.x >> 16, x[2], x[3]);
    widen_e4m3x2(w.y, x[4], x[5]);
    widen_e4m3x2(w.y >> 16, x[6], x[7]);
  } else if constexpr (DPL == 4) {
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(src));
    widen_e4m3x2(w, x[0], x[1]);
    widen_e4m3x2(w >> 16, x[2], x[3]);
  } else {
    const uint32_t w = __ldg(reinterpret_cast<const uint16_t*>(src));
    widen_e4m3x2(w, x[0], x[1]);
  }
}

// Keys of split s of a sequence of length Sk: [s*per, min(Sk, (s+1)*per)) with
// per = ceil(ceil(Sk / splits) / 16) * 16.
__device__ __forceinline__ void split_range(int Sk, int splits, int s, int& k0, int& k1) {
  int per = (Sk + splits - 1) / splits;
  per = (per + 15) / 16 * 16;
  k0 = min(Sk, s * per);
  k1 = min(Sk, k0 + per);
}

template <bool BF16>
__device__ __forceinline__ void store_out(void* out, int64_t idx, const float* v, int n, int mode) {
  if (mode == 3) {
    float* o = static_cast<float*>(out) + idx;
    for (int e = 0; e < n; ++e) o[e] = v[e];
  } else {
    uint16_t* o = static_cast<uint16_t*>(out) + idx;
    for (int e = 0; e < n; ++e) o[e] = round_out<BF16>(v[e], mode);
  }
}

template <int D, bool BF16, int GH, bool KV8>
__global__ void __launch_bounds__(kDecWarps * 32) decode_split_kernel(const __grid_constant__ DecodeParams p) {
  using KvT = std::conditional_t<KV8, uint8_t, uint16_t>;   // cache element (fp8 code or 16-bit)
  constexpr int DPL = D / 32;             // channels per lane
  constexpr int CK = (GH <= 4 && D <= 128) ? 16 : 8;    // keys per chunk
  constexpr int N = CK * GH;              // dot products per chunk
  constexpr int NV = N >= 32 ? N / 32 : 1;

  __shared__ float s_sc[kDecWarps][CK][GH];
  __shared__ float s_m[kDecWarps][GH];
  __shared__ float s_l[kDecWarps][GH];
  __shared__ float s_a[kDecWarps][GH];
  __shared__ float s_o[kDecWarps][GH][D];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int hg = blockIdx.y;
  const int b = blockIdx.z;
  const int G = p.num_q_heads / p.num_kv_heads;
  const int h0 = hg * GH;
  const int kvh = h0 / G;
  const int Sk = p.seq_lens[b];
  if (Sk < 0 || Sk > p.max_seqlen_k) {
    if (threadIdx.x == 0 && split == 0 && hg == 0) report_status(p.status, kStatusBadArg);
    return;
  }
  // A sliding window keeps keys >= lo (the decode row's aligned key is
  // Sk - 1); the splits cut [lo rounded down to 16, Sk) and keys below lo
  // are masked, so chunks stay page-aligned.
  const int lo = p.win_left >= 0 ? max(0, Sk - 1 - p.win_left) : 0;
  const int lo16 = lo & ~15;
  int k_begin, k_end;
  split_range(Sk - lo16, p.num_splits, split, k_begin, k_end);
  k_begin += lo16;
  k_end += lo16;
  const float inv_cap = p.softcap > 0.f ? 1.f / p.softcap : 0.f;

  const uint16_t* qb =
      static_cast<const uint16_t*>(p.q) + ((int64_t)b * p.num_q_heads + h0) * D + lane * DPL;
  float q[GH][DPL];
#pragma unroll
  for (int h = 0; h < GH; ++h) load_row<BF16, DPL>(qb + h * D, q[h]);

  float o[GH][DPL];
#pragma unroll
  for (int h = 0; h < GH; ++h)
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[h][e] = 0.f;
  if (lane < GH) {
    s_m[warp][lane] = -INFINITY;
    s_l[warp][lane] = 0.f;
  }
  __syncwarp();

  const int bs = p.block_size;
  const int32_t* bt = p.block_table + (int64_t)b * p.bt_stride;
  const int64_t slot_stride = (int64_t)p.num_kv_heads * D;  // elements between consecutive slots
  const KvT* kc = static_cast<const KvT*>(p.k_cache);
  const KvT* vc = static_cast<const KvT*>(p.v_cache);
  const float sl2 = p.scale_log2;

  for (int k0 = k_begin + warp * CK; k0 < k_end; k0 += kDecWarps * CK) {
    const int nv = min(CK, k_end - k0);
    const int page = bt[k0 / bs];
    if (page < 0 || page >= p.num_blocks) {
      if (lane == 0) report_status(p.status, kStatusBadBlockTable);
      continue;
    }
    const int64_t base = ((int64_t)page * bs + (k0 % bs)) * slot_stride + (int64_t)kvh * D + lane * DPL;

    // ---- dot products q_h . K_r for the chunk
    float kx[CK][DPL];
#pragma unroll
    for (int r = 0; r < CK; ++r) {
      if (r < nv) {
        if constexpr (KV8) load_row8<DPL>(kc + base + r * slot_stride, kx[r]);
        else load_row<BF16, DPL>(kc + base + r * slot_stride, kx[r]);
      }
      else
#pragma unroll
        for (int e = 0; e < DPL; ++e) kx[r][e] = 0.f;
    }
    float part[N];
#pragma unroll
    for (int r = 0; r < CK; ++r)
#pragma unroll
      for (int h = 0; h < GH; ++h) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc = fmaf(q[h][e], kx[r][e], acc);
        part[r * GH + h] = acc;
      }
    scatter_step<N, N, 16>(part, lane);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int idx = scatter_index<N>(lane, k);
      const int r = idx / GH, h = idx % GH;
      float sc = part[k] * sl2;
      if (p.score_xform) {
        // softcap / ALiBi on the scaled score, distance to the last key
        const float slope = p.alibi ? p.alibi[h0 + h] : 0.f;
        const float x = rewrite_score(part[k] * p.scale, p.softcap, inv_cap, slope,
                                      (float)(Sk - 1 - (k0 + r)));
        sc = x * 1.4426950408889634f;
      }
      s_sc[warp][r][h] = (r < nv && k0 + r >= lo) ? sc : -INFINITY;
    }
    __syncwarp();

    // ---- online softmax bookkeeping, one lane per head
    if (lane < GH) {
      const int h = lane;
      float cm = -INFINITY;
#pragma unroll
      for (int r = 0; r < CK; ++r) cm = fmaxf(cm, s_sc[warp][r][h]);
      const float m_old = s_m[warp][h];
      const float m_new = fmaxf(m_old, cm);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float a = fast_exp2(m_old - m_use);
      float l = s_l[warp][h] * a;
#pragma unroll
      for (int r = 0; r < CK; ++r) {
        const float pr = fast_exp2(s_sc[warp][r][h] - m_use);
        s_sc[warp][r][h] = pr;
        l += pr;
      }
      s_l[warp][h] = l;
      s_m[warp][h] = m_new;
      s_a[warp][h] = a;
    }
    __syncwarp();

    // ---- o = alpha * o + sum_r p_r V_r
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      const float a = s_a[warp][h];
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[h][e] *= a;
    }
    float vx[CK][DPL];
#pragma unroll
    for (int r = 0; r < CK; ++r) {
      if (r < nv) {
        if constexpr (KV8) load_row8<DPL>(vc + base + r * slot_stride, vx[r]);
        else load_row<BF16, DPL>(vc + base + r * slot_stride, vx[r]);
      }
      else
#pragma unroll
        for (int e = 0; e < DPL; ++e) vx[r][e] = 0.f;
    }
#pragma unroll
    for (int r = 0; r < CK; ++r) {
      if (r < nv) {
#pragma unroll
        for (int h = 0; h < GH; ++h) {
          const float pr = s_sc[warp][r][h];
#pragma unroll
          for (int e = 0; e < DPL; ++e) o[h][e] = fmaf(pr, vx[r][e], o[h][e]);
        }
      }
    }
    __syncwarp();
  }

  // ---- merge the warps' states in a fixed order
#pragma unroll
  for (int h = 0; h < GH; ++h)
#pragma unroll
    for (int e = 0; e < DPL; ++e) s_o[warp][h][lane * DPL + e] = o[h][e];
  __syncthreads();

  const int Hq = p.num_q_heads;
  for (int idx = threadIdx.x; idx < GH * D; idx += kDecWarps * 32) {
    const int h = idx / D, e = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, s_m[w][h]);
    const float Mu = M == -INFINITY ? 0.f : M;
    float acc = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      const float wgt = fast_exp2(s_m[w][h] - Mu);
      acc = fmaf(wgt, s_o[w][h][e], acc);
      L = fmaf(wgt, s_l[w][h], L);
    }
    const int64_t row = (int64_t)b * Hq + h0 + h;
    if (p.num_splits == 1) {
      float v, lse_v;
      if (p.sinks) {
        // the sink term joins the denominator here
        float inv_l;
        finish_row(M, L, p.sinks[h0 + h], inv_l, lse_v);
        v = acc * inv_l;
      } else {
        // L == 0: no visible key; a NaN L (a NaN score) stays NaN
        v = L != 0.f ? acc / L : 0.f;
        lse_v = L != 0.f ? M * kLn2 + logf(L) : -INFINITY;
      }
      v *= p.out_scale;   // fp8 V factor (1 otherwise)
      store_out<BF16>(p.out, row * D + e, &v, 1, p.rounding);
      if (e == 0 && p.lse) p.lse[row] = lse_v;
    } else {
      p.part_o[(row * p.num_splits + split) * D + e] = acc;
      if (e == 0) {
        p.part_ml[(row * p.num_splits + split) * 2 + 0] = M;
        p.part_ml[(row * p.num_splits + split) * 2 + 1] = L;
      }
    }
  }
}

// Log-sum-exp merge of the split partials: with lse_p = m_p + ln l_p the
// result is sum_p e^(lse_p - lse*) (o_p / l_p) / sum_p e^(lse_p - lse*); since
// (o_p / l_p) e^(lse_p) = o_p e^(m_p), this is computed as
// sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p with M = max_p m_p (m in log2
// units), summed in split order.  One warp per (sequence, q head).
template <int D, bool BF16>
__global__ void __launch_bounds__(128) decode_combine_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int DPL = D / 32;                   // channels per lane: 8, 4 or 2 at d = 256, 128, 64
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= (int64_t)p.num_seqs * p.num_q_heads) return;
  const int S = p.num_splits;                   // at most 64
  // Lane s holds the (m, l) of split s and of split s + 32: one memory round
  // trip for all of them; the max and the weight sum are warp reductions
  // (every lane ends with the same values).
  const float* ml = p.part_ml + row * S * 2;
  float m_a = -INFINITY, l_a = 0.f, m_b = -INFINITY, l_b = 0.f;
  if (lane < S) {
    const float2 v = *reinterpret_cast<const float2*>(ml + 2 * lane);
    m_a = v.x;
    l_a = v.y;
  }
  if (lane + 32 < S) {
    const float2 v = *reinterpret_cast<const float2*>(ml + 2 * (lane + 32));
    m_b = v.x;
    l_b = v.y;
  }
  float M = fmaxf(m_a, m_b);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
  const float Mu = M == -INFINITY ? 0.f : M;
  const float w_a = fast_exp2(m_a - Mu), w_b = fast_exp2(m_b - Mu);   // 0 for empty splits
  float L = w_a * l_a + w_b * l_b;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xFFFFFFFFu, L, o);
  // The partial rows, eight splits' loads in flight at a time, accumulated
  // in split order.
  float acc[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
  const float* po = p.part_o + row * S * D + lane * DPL;
  for (int s0 = 0; s0 < S; s0 += 8) {
    float v[8][DPL];
    float wg[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int sp = s0 + u;
      const float w = __shfl_sync(0xFFFFFFFFu, sp < 32 ? w_a : w_b, sp & 31);
      wg[u] = sp < S ? w : 0.f;
      if (sp < S) {
        if constexpr (DPL % 4 == 0) {
#pragma unroll
          for (int q4 = 0; q4 < DPL / 4; ++q4) {
            const float4 x = *reinterpret_cast<const float4*>(po + (int64_t)sp * D + 4 * q4);
            v[u][4 * q4] = x.x; v[u][4 * q4 + 1] = x.y; v[u][4 * q4 + 2] = x.z; v[u][4 * q4 + 3] = x.w;
          }
        } else {
          const float2 x = *reinterpret_cast<const float2*>(po + (int64_t)sp * D);
          v[u][0] = x.x; v[u][1] = x.y;
        }
      } else {
#pragma unroll
        for (int e = 0; e < DPL; ++e) v[u][e] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[e] = fmaf(wg[u], v[u][e], acc[e]);
  }
  // the weights are relative to 2^Mu: the merged state is (m, l) = (Mu, L),
  // plus the sink term when the call has one
  float inv, lse_v;
  finish_row(M == -INFINITY ? -INFINITY : Mu, L, p.sinks ? p.sinks[row % p.num_q_heads] : -INFINITY,
             inv, lse_v);
  inv *= p.out_scale;   // fp8 V factor (1 otherwise)
#pragma unroll
  for (int e = 0; e < DPL; ++e) acc[e] *= inv;
  store_out<BF16>(p.out, row * D + lane * DPL, acc, DPL, p.rounding);
  if (lane == 0 && p.lse) p.lse[row] = lse_v;
}

template <int D, bool BF16>
cudaError_t launch_combine_t(const DecodeParams& p, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.num_seqs * p.num_q_heads;
  decode_combine_kernel<D, BF16><<<(unsigned)((rows + 3) / 4), 128, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int D, bool BF16, int GH>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t stream) {
  const int G = p.num_q_heads / p.num_kv_heads;
  dim3 grid(p.num_splits, p.num_kv_heads * (G / GH), p.num_seqs);
  if (p.kv_fp8) decode_split_kernel<D, BF16, GH, true><<<grid, kDecWarps * 32, 0, stream>>>(p);
  else decode_split_kernel<D, BF16, GH, false><<<grid, kDecWarps * 32, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.num_splits == 1) return e;
  return launch_combine_t<D, BF16>(p, stream);
}

template <int D, bool BF16>
cudaError_t launch_decode_d(const DecodeParams& p, int gh, cudaStream_t stream) {
  switch (gh) {
    case 1: return launch_decode_t<D, BF16, 1>(p, stream);
    case 2: return launch_decode_t<D, BF16, 2>(p, stream);
    case 4: return launch_decode_t<D, BF16, 4>(p, stream);
    case 8:
      if constexpr (D <= 128) return launch_decode_t<D, BF16, 8>(p, stream);
      else return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

__global__ void round_kernel(void* out, const float* in, int64_t n, int bf16, int mode) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float x = in[i];
    static_cast<uint16_t*>(out)[i] = bf16 ? round_out<true>(x, mode) : round_out<false>(x, mode);
  }
}

}  // namespace

// Heads handled per CTA: the largest of 8, 4, 2, 1 that divides the group
// (at most 4 at head size 256, whose per-warp partial rows would otherwise
// exceed the static shared memory of a CTA).
static int heads_per_cta(int group, int head_size) {
  for (int gh = head_size == 256 ? 4 : 8; gh > 1; gh >>= 1)
    if (group % gh == 0) return gh;
  return 1;
}

cudaError_t launch_decode(const DecodeParams& p, int head_size, bool bf16, int group,
                          cudaStream_t stream) {
  const int gh = heads_per_cta(group, head_size);
  if (head_size == 256) return bf16 ? launch_decode_d<256, true>(p, gh, stream) : launch_decode_d<256, false>(p, gh, stream);
  if (head_size == 128) return bf16 ? launch_decode_d<128, true>(p, gh, stream) : launch_decode_d<128, false>(p, gh, stream);
  if (head_size == 64) return bf16 ? launch_decode_d<64, true>(p, gh, stream) : launch_decode_d<64, false>(p, gh, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_combine(const DecodeParams& p, int head_size, bool bf16,
                                  cudaStream_t stream) {
  if (head_size == 256) return bf16 ? launch_combine_t<256, true>(p, stream) : launch_combine_t<256, false>(p, stream);
  if (head_size == 128) return bf16 ? launch_combine_t<128, true>(p, stream) : launch_combine_t<128, false>(p, stream);
  if (head_size == 64) return bf16 ? launch_combine_t<64, true>(p, stream) : launch_combine_t<64, false>(p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_round(void* out, const float* in, int64_t n, bool bf16, int mode,
                         cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 152 * 16);
  round_kernel<<<(unsigned)blocks, 256, 0, stream>>>(out, in, n, bf16 ? 1 : 0, mode);
  return cudaGetLastError();
}

}  // namespace attn

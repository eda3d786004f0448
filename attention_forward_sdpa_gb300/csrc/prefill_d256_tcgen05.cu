// prefill_d256_tcgen05.cu -- the fused SDPA forward of prefill_tcgen05.cu for
// head size 256 ("gfx942 unified attention, from the math up": the same
// online-softmax recurrence of sec. 3, the bottom-right causal mask and early
// exit of sec. 4 and the paged cache of sec. 5; the pages leave d = 256
// without a tiled kernel).
//
// At d = 256 one query tile's fp32 accumulator O (128 x 256) takes half of the
// 512 tensor-memory columns, so a CTA owns ONE 128-row query tile and keeps
// two score buffers instead of two query tiles: S(j+1) is computed while the
// softmax works on S(j), and the tensor pipe alternates P(j) V_j with
// Q K_{j+2}^T.  TMEM map (columns): S_a [0,128), S_b [128,256), O [256,512);
// P(j) overwrites the first 64 columns of its score buffer as packed 16-bit
// pairs and is the A operand of P V.
//
// Shared memory: Q (128 x 256, 64 KB, four 128-byte-swizzled column blocks)
// and a ring of five 32 KB slots.  A 128-key K tile fills two slots (channels
// 0-127, 128-255: the two halves of the Q K^T contraction); a V tile fills two
// slots (keys 0-63, 64-127: the two halves of the P V contraction).  The
// producer fills the slots in the order the MMA thread consumes them:
// K_0, K_1, then per key tile j: V_j, K_{j+2}.
//
// Warp roles: warp 0 TMA producer (one thread), warp 1 TMEM owner and MMA
// issuer (one thread), warps 4-7 softmax and epilogue (one thread per query
// row; warps 2-3 only take part in the CTA barriers).  With the score buffers
// in flight ahead of P V, the product P(j-1) V_{j-1} may still be running when
// the softmax of tile j finds that the running max moved; it then waits for
// that product (a per-product barrier) before rescaling O.  Every pipeline
// wait is bounded; one that runs out raises the CTA's abort flag and the
// status word records ATTN_ERR_TIMEOUT.

#include "attn_internal.h"
#include "round16.cuh"
#include "score_features.cuh"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kD = 256;
constexpr int kBM = 128;                 // query rows per tile
constexpr int kBN = 128;                 // keys per KV tile
constexpr int kThreads = 256;            // 8 warps
constexpr int kSlots = 5;                // ring slots
constexpr int kSlotBytes = 32768;
constexpr int kQBytes = kBM * kD * 2;    // 64 KB
constexpr int kColBlock = 16384;         // 128 rows x 128 bytes: one swizzled column block of Q or K
constexpr int kVBlock = 8192;            // 64 rows x 128 bytes: one column block of a V slot
constexpr int kRingOff = kQBytes;
constexpr int kBarOff = kRingOff + kSlots * kSlotBytes;
// q_full, slot_full[5], slot_empty[5], s_full[2], p_full[2], pv_done, o_full, mma_done
constexpr int kNumBars = 1 + 2 * kSlots + 2 + 2 + 3;
constexpr int kMiscOff = kBarOff + kNumBars * 8;
constexpr int kSmemBytes = kMiscOff + 16 + 1024;   // + slack for the 1024-byte alignment
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 256;
constexpr float kRescaleSlack = 8.f;     // log2 units: p stays <= 256

static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) break;
  }
}

// min(a, b + c) without int32 overflow (window bounds may be huge)
__device__ __forceinline__ int min_sum(int a, int b, int c) {
  const long long v = (long long)b + (long long)c;
  return v < (long long)a ? (int)v : a;
}

// FEAT: the feature-flagged instantiation (sliding window, score rewrite,
// sinks); without it the flags are compile-time off.
template <bool BF16, bool FEAT>
__global__ void __launch_bounds__(kThreads, 1) prefill_d256_kernel(const __grid_constant__ PrefillParams p) {
  const int win_left = FEAT ? p.win_left : -1;
  const int win_right = FEAT ? p.win_right : -1;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sRing = base + kRingOff;
  const uint32_t bars = base + kBarOff;
  const uint32_t bar_q_full = bars;
  const uint32_t bar_full = bars + 8u;                          // [kSlots]
  const uint32_t bar_empty = bar_full + 8u * kSlots;            // [kSlots]
  const uint32_t bar_s_full = bar_empty + 8u * kSlots;          // [2]
  const uint32_t bar_p_full = bar_s_full + 16u;                 // [2]
  const uint32_t bar_pv_done = bar_p_full + 16u;
  const uint32_t bar_o_full = bar_pv_done + 8u;
  const uint32_t bar_mma_done = bar_o_full + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ------------------------------------------------------------ work item
  const int b = blockIdx.y;
  int q_begin = 0, Sq = p.dense_sq, Sk = p.dense_sk;
  if (!p.dense) {
    q_begin = p.query_start_loc[b];
    const int q_end = p.query_start_loc[b + 1];
    Sq = q_end - q_begin;
    Sk = p.seq_lens[b];
    if (q_begin < 0 || Sq < 0 || Sq > p.max_seqlen_q || q_end > p.total_q || Sk < 0 ||
        Sk > p.max_seqlen_k) {
      if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0) report_status(p.status, kStatusBadArg);
      return;
    }
  }
  const int n_rb = (Sq + kBM - 1) / kBM;
  if ((int)blockIdx.z >= n_rb) return;
  const int row0 = (n_rb - 1 - (int)blockIdx.z) * kBM;   // heaviest (last) row block first
  const int head = blockIdx.x;
  const int rows = min(kBM, Sq - row0);
  const int off = Sk - Sq;                                // row i sees keys j <= i + off
  const int last = row0 + rows - 1;
  // keys [lo, lim) of the tile's rows: the causal bound and a sliding window
  // narrow them; lim_lo is the smallest upper limit and lo_hi the largest
  // lower limit (tiles past lim_lo or before lo_hi need the element mask)
  int lim = Sk, lim_lo = Sk, lo_first = 0, lo_hi = 0;
  if (p.causal) {
    lim = min(lim, last + off + 1);
    lim_lo = min(lim_lo, row0 + off + 1);
  }
  if (win_right >= 0) {
    lim = min_sum(lim, last + off + 1, win_right);
    lim_lo = min_sum(lim_lo, row0 + off + 1, win_right);
  }
  if (win_left >= 0) {
    lo_first = max(0, row0 + off - win_left);
    lo_hi = max(0, last + off - win_left);
  }
  const int j0 = FEAT ? lo_first / kBN : 0;   // first key tile; tiles before it are skipped
  const int nkv = lim > lo_first ? (lim + kBN - 1) / kBN - j0 : 0;   // key tiles from j0
  const int kvh = head / (p.num_q_heads / p.num_kv_heads);

  // ------------------------------------------------------------ setup
  if (threadIdx.x == 0) {
    mbar_init(bar_q_full, 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar_full + 8u * s, 1);
      mbar_init(bar_empty + 8u * s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_s_full + 8u * t, 1);
      mbar_init(bar_p_full + 8u * t, kBM);
    }
    mbar_init(bar_pv_done, 1);
    mbar_init(bar_o_full, 1);
    mbar_init(bar_mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0 && !p.stall_producer && nkv > 0) {
      mbar_arrive_expect_tx(bar_q_full, kQBytes);
      for (int c = 0; c < 4; ++c) {
        if (p.dense) tma_load_4d(sQ + c * kColBlock, &p.tm_q, bar_q_full, c * 64, head, row0, b);
        else tma_load_3d(sQ + c * kColBlock, &p.tm_q, bar_q_full, c * 64, head, q_begin + row0);
      }
      const int bs = p.block_size;
      const int n_pages = (Sk + bs - 1) / bs;
      const int32_t* bt = p.block_table + (int64_t)b * p.bt_stride;
      int filled[kSlots];
#pragma unroll
      for (int s = 0; s < kSlots; ++s) filled[s] = 0;
      int pos = 0;
      bool ok = true;
      // claims the next ring slot; returns its shared address and barrier
      auto claim = [&](uint32_t& dst, uint32_t& bar) -> bool {
        const int s = pos % kSlots, u = pos / kSlots;
        ++pos;
        if (u > 0 && !mbar_wait(bar_empty + 8u * s, (u - 1) & 1, abort_flag, p.wait_limit_ns)) return false;
        filled[s] = u + 1;
        dst = sRing + s * kSlotBytes;
        bar = bar_full + 8u * s;
        return true;
      };
      // K_j, channels [128 h, 128 h + 128): column blocks 2h, 2h+1 of 128 keys
      auto load_k = [&](int j, int h) -> bool {
        uint32_t dst, bar;
        if (!claim(dst, bar)) return false;
        const int key0 = j * kBN;
        if (bs >= kBN) {
          const int page = p.dense ? b : bt[key0 / bs];
          if (page < 0 || page >= p.num_blocks) report_status(p.status, kStatusBadBlockTable);
          mbar_arrive_expect_tx(bar, kSlotBytes);
          for (int c = 0; c < 2; ++c)
            tma_load_4d(dst + c * kColBlock, &p.tm_k, bar, (2 * h + c) * 64, kvh, key0 % bs, page);
        } else {
          const int first = key0 / bs;
          const int cnt = min(kBN / bs, n_pages - first);
          mbar_arrive_expect_tx(bar, (uint32_t)(cnt * 2 * bs * 128));
          for (int r = 0; r < cnt; ++r) {
            const int page = bt[first + r];
            if (page < 0 || page >= p.num_blocks) report_status(p.status, kStatusBadBlockTable);
            for (int c = 0; c < 2; ++c)
              tma_load_4d(dst + c * kColBlock + r * bs * 128, &p.tm_k, bar, (2 * h + c) * 64, kvh, 0, page);
          }
        }
        return true;
      };
      // V_j, keys [64 h, 64 h + 64) of the tile: four column blocks of 64 rows
      auto load_v = [&](int j, int h) -> bool {
        uint32_t dst, bar;
        if (!claim(dst, bar)) return false;
        const int key0 = j * kBN + 64 * h;
        if (bs >= 64) {
          const int pg = key0 / bs;
          if (!p.dense && pg >= n_pages) {
            mbar_arrive_expect_tx(bar, 0);   // no key of this half exists: nothing to copy
            return true;
          }
          const int page = p.dense ? b : bt[pg];
          if (page < 0 || page >= p.num_blocks) report_status(p.status, kStatusBadBlockTable);
          mbar_arrive_expect_tx(bar, kSlotBytes);
          for (int c = 0; c < 4; ++c)
            tma_load_4d(dst + c * kVBlock, &p.tm_v, bar, c * 64, kvh, key0 % bs, page);
        } else {
          const int first = key0 / bs;
          const int cnt = max(0, min(64 / bs, n_pages - first));
          mbar_arrive_expect_tx(bar, (uint32_t)(cnt * 4 * bs * 128));
          for (int r = 0; r < cnt; ++r) {
            const int page = bt[first + r];
            if (page < 0 || page >= p.num_blocks) report_status(p.status, kStatusBadBlockTable);
            for (int c = 0; c < 4; ++c)
              tma_load_4d(dst + c * kVBlock + r * bs * 128, &p.tm_v, bar, c * 64, kvh, 0, page);
          }
        }
        return true;
      };
      for (int j = 0; ok && j < min(nkv, 2); ++j) ok = load_k(j0 + j, 0) && load_k(j0 + j, 1);
      for (int j = 0; ok && j < nkv; ++j) {
        ok = load_v(j0 + j, 0) && load_v(j0 + j, 1);
        if (ok && j + 2 < nkv) ok = load_k(j0 + j + 2, 0) && load_k(j0 + j + 2, 1);
      }
      // make sure no copy into this CTA's shared memory is still in flight
      for (int s = 0; s < kSlots; ++s)
        if (filled[s] > 0) drain_wait(bar_full + 8u * s, (filled[s] - 1) & 1, p.wait_limit_ns);
      drain_wait(bar_q_full, 0, p.wait_limit_ns);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------- MMA issuer
    const uint32_t idesc_s = make_idesc_f16(BF16, kBM, kBN, false);
    const uint32_t idesc_pv = make_idesc_f16(BF16, kBM, kD, true);
    const uint64_t dq = make_sdesc_sw128(sQ, 16, 1024);            // Q, K-major
    const uint64_t dk = make_sdesc_sw128(sRing, 16, 1024);         // K half in slot 0, K-major
    const uint64_t dv = make_sdesc_sw128(sRing, kVBlock, 1024);    // V half in slot 0, MN-major
    constexpr uint64_t kSlotStep = kSlotBytes >> 4;
    int pos = 0;
    bool ok = true;
    auto take = [&](int& slot) -> bool {
      slot = pos % kSlots;
      const int u = pos / kSlots;
      ++pos;
      if (!mbar_wait(bar_full + 8u * slot, u & 1, abort_flag, p.wait_limit_ns)) return false;
      tc_fence_after();
      return true;
    };
    // S_buf (+)= Q[:, 128h : 128h+128] K_j[:, 128h : 128h+128]^T, 8 K-steps
    auto issue_s_half = [&](int buf, int h, int slot) {
      const uint64_t kb = dk + (uint64_t)slot * kSlotStep;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int ka = 8 * h + kk;
        const uint64_t ao = (uint64_t)(((ka >> 2) * kColBlock + (ka & 3) * 32) >> 4);
        const uint64_t bo = (uint64_t)((((kk >> 2) & 1) * kColBlock + (kk & 3) * 32) >> 4);
        umma_ss(tmem + 128u * buf, dq + ao, kb + bo, idesc_s, ka > 0 ? 1u : 0u);
      }
    };
    // O (+)= P_buf[:, 64h : 64h+64] V_j[64h : 64h+64, :], 4 K-steps of 16 keys
    auto issue_pv_half = [&](int buf, int h, int slot, bool acc) {
      const uint64_t vb = dv + (uint64_t)slot * kSlotStep;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int kg = 4 * h + kk;
        umma_ts(tmem + kOCol, tmem + 128u * buf + kg * 8, vb + (uint64_t)((kk * 16 * 128) >> 4), idesc_pv,
                (acc || kg > 0) ? 1u : 0u);
      }
    };
    // S(j) into buffer j & 1: both channel halves of K_j
    auto issue_s = [&](int j) -> bool {
      for (int h = 0; h < 2; ++h) {
        int slot;
        if (!take(slot)) return false;
        issue_s_half(j & 1, h, slot);
        umma_commit(bar_empty + 8u * slot);
      }
      umma_commit(bar_s_full + 8u * (j & 1));
      return true;
    };
    if (nkv > 0) ok = mbar_wait(bar_q_full, 0, abort_flag, p.wait_limit_ns);
    for (int j = 0; ok && j < min(nkv, 2); ++j) ok = issue_s(j);
    for (int j = 0; ok && j < nkv; ++j) {
      const int buf = j & 1;
      if (!mbar_wait(bar_p_full + 8u * buf, (j >> 1) & 1, abort_flag, p.wait_limit_ns)) break;
      tc_fence_after();
      for (int h = 0; ok && h < 2; ++h) {
        int slot;
        if (!take(slot)) { ok = false; break; }
        const int r0 = Sk - ((j0 + j) * kBN + 64 * h);   // rows >= r0 of this half lie past kv_len
        if (r0 < 64) {
          // their V rows may hold anything (NaN included); P is 0 there but
          // 0 * NaN is not, so zero them
          uint8_t* vt = smem + kRingOff + slot * kSlotBytes;
          const int first = max(r0, 0);
          for (int idx = 0; idx < (64 - first) * 4 * 8; ++idx) {
            const int chunk = idx & 7;
            const int c = (idx >> 3) & 3;
            const int r = first + (idx >> 5);
            *reinterpret_cast<uint4*>(vt + c * kVBlock + r * 128 + chunk * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        issue_pv_half(buf, h, slot, j > 0);
        umma_commit(bar_empty + 8u * slot);
      }
      if (!ok) break;
      umma_commit(bar_pv_done);
      if (j + 1 == nkv) umma_commit(bar_o_full);
      if (j + 2 < nkv) ok = issue_s(j + 2);
    }
    // no MMA may still be running when TMEM is released
    umma_commit(bar_mma_done);
    drain_wait(bar_mma_done, 0, p.wait_limit_ns);
  } else if (warp >= 4) {
    // ---------------------------------------------------------- softmax + epilogue
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tO = tmem + lane_off + kOCol;
    const int i_row = row0 + r;
    int key_lim = p.causal ? min(Sk, i_row + off + 1) : Sk;
    if (win_right >= 0) key_lim = min_sum(key_lim, i_row + off + 1, win_right);
    const int key_lo = win_left >= 0 ? i_row + off - win_left : 0;
    const float sl2 = p.scale_log2;
    const float slope = FEAT && p.alibi ? p.alibi[head] : 0.f;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int buf = j & 1;
      const int jk = j0 + j;                 // key tile
      const uint32_t tS = tmem + lane_off + 128u * buf;
      if (!mbar_wait(bar_s_full + 8u * buf, (j >> 1) & 1, abort_flag, p.wait_limit_ns)) { ok = false; break; }
      tc_fence_after();
      uint32_t s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, s[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait(s[c]);
      if (FEAT && p.score_xform) rewrite_scores(s, p.scale, p.softcap, slope, (float)(i_row + off - jk * kBN));
      if ((jk + 1) * kBN > lim_lo || (FEAT && jk * kBN < lo_hi)) {
        const int cl = key_lim - jk * kBN;  // columns >= cl are masked for this row
        const int cf = key_lo - jk * kBN;   // and columns < cf
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (32 * c + e >= cl || (FEAT && 32 * c + e < cf)) s[c][e] = 0xFF800000u;  // -inf
      }
      float mc[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) mc[c] = __uint_as_float(s[c][0]);
#pragma unroll
      for (int i = 1; i + 1 < 32; i += 2)
#pragma unroll
        for (int c = 0; c < 4; ++c)
          mc[c] = fmax3(mc[c], __uint_as_float(s[c][i]), __uint_as_float(s[c][i + 1]));
      const float mx = fmax3(fmaxf(mc[0], __uint_as_float(s[0][31])), fmaxf(mc[1], __uint_as_float(s[1][31])),
                             fmax3(mc[2], mc[3], fmaxf(__uint_as_float(s[2][31]), __uint_as_float(s[3][31]))));
      // lazy running max (exact: o and l share the reference value)
      const float mxs = mx * sl2;
      const float m_new = (mxs > m + kRescaleSlack) ? mxs : m;
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = fast_exp2(m - m_use);
      const float2 sc2 = make_float2(sl2, sl2);
      const float2 nm2 = make_float2(-m_use, -m_use);
      float2 rs[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) rs[a] = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 x = ffma2(make_float2(__uint_as_float(s[c][2 * e]), __uint_as_float(s[c][2 * e + 1])),
                                 sc2, nm2);
          const float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
          rs[e & 3] = fadd2(rs[e & 3], pp);
          pk[e] = BF16 ? pack_bf16x2_rn(pp.x, pp.y) : pack_f16x2_rn(pp.x, pp.y);
        }
        tmem_st16(tS + 16 * c, pk);
      }
      if (j > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
        // O must hold P(j-1) V_{j-1} before it is rescaled: that product was
        // issued after S(j) and may still be running.
        if (!mbar_wait(bar_pv_done, (j - 1) & 1, abort_flag, p.wait_limit_ns)) { ok = false; break; }
        tc_fence_after();
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 2
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * c, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 v = fmul2(make_float2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), a2);
            o[2 * e] = __float_as_uint(v.x);
            o[2 * e + 1] = __float_as_uint(v.y);
          }
          tmem_st32(tO + 32 * c, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p_full + 8u * buf);
      const float2 r01 = fadd2(rs[0], rs[1]), r23 = fadd2(rs[2], rs[3]);
      l = l * alpha + ((r01.x + r23.x) + (r01.y + r23.y));
      m = m_new;
    }
    if (ok && nkv > 0) {
      ok = mbar_wait(bar_o_full, 0, abort_flag, p.wait_limit_ns);
      tc_fence_after();
    }
    const bool row_ok = r < rows;
    const int64_t tok = (int64_t)q_begin + row0 + r;
    float inv_l, lse_v;
    finish_row(m, l, FEAT && p.sinks ? p.sinks[head] : -INFINITY, inv_l, lse_v);
    if (FEAT) inv_l *= p.out_scale;   // fp8 V factor (1 otherwise)
    // The Q buffer is free once o_full has fired (it covers every product
    // that read Q); the epilogue stages its output there.
    if (rows == kBM && p.rounding != 3) {
      // full tile, 16-bit output: swizzled rows in the Q buffer, one TMA store
      if (ok) {
#pragma unroll 1
        for (int c2 = 0; c2 < kD / 64; ++c2) {
          uint32_t o[2][32];
          if (nkv > 0) {
            tmem_ld32(tO + 64 * c2, o[0]);
            tmem_ld32(tO + 64 * c2 + 32, o[1]);
            tmem_ld_wait(o[0]);
            tmem_ld_wait(o[1]);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[0][e] = o[1][e] = 0u;
          }
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {
            uint32_t w[16];
            round_pack32<BF16>(o[hc], inv_l, p.rounding, w);
            uint8_t* rowp = smem + c2 * kColBlock + r * 128;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int chunk = hc * 4 + v;
              *reinterpret_cast<uint4*>(rowp + ((chunk ^ (r & 7)) * 16)) =
                  make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
            }
          }
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, kBM);
      if (wq == 0 && lane == 0 && ok && *abort_flag == 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (p.dense) tma_store_4d(&p.tm_o, sQ + c * kColBlock, c * 64, head, row0, b);
          else tma_store_3d(&p.tm_o, sQ + c * kColBlock, c * 64, head, q_begin + row0);
        }
        bulk_commit_group();
        bulk_wait_group_read0();
      }
    } else if (ok) {
      // 64 bytes of each of the warp's 32 rows at a time through a 2 KB
      // staging buffer (pieces rotated by row to spread the banks)
      uint8_t* stage = smem + wq * 2048;
      const int64_t row_elems = p.dense ? p.o_stride_s : (int64_t)p.num_q_heads * kD;
      const int64_t tile_base =
          p.dense ? (int64_t)b * p.o_stride_b + (int64_t)(row0 + wq * 32) * p.o_stride_s +
                        (int64_t)head * p.o_stride_h
                  : ((int64_t)q_begin + row0 + wq * 32) * row_elems + (int64_t)head * kD;
      const int rows_here = min(32, rows - wq * 32);
      auto flush = [&](int64_t col_byte) {
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int rr = 8 * k + (lane >> 2), piece = lane & 3;
          const uint4 v = *reinterpret_cast<const uint4*>(stage + rr * 64 + ((piece ^ (rr & 3)) * 16));
          if (rr < rows_here) {
            uint8_t* g = reinterpret_cast<uint8_t*>(p.out) +
                         (tile_base + (int64_t)rr * row_elems) * (p.rounding == 3 ? 4 : 2) + col_byte +
                         piece * 16;
            *reinterpret_cast<uint4*>(g) = v;
          }
        }
        __syncwarp();
      };
#pragma unroll 1
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t o[32];
        if (nkv > 0) {
          tmem_ld32(tO + 32 * c, o);
          tmem_ld_wait(o);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (p.rounding == 3) {
#pragma unroll
          for (int hlf = 0; hlf < 2; ++hlf) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              *reinterpret_cast<float4*>(stage + lane * 64 + ((v ^ (lane & 3)) * 16)) =
                  make_float4(__uint_as_float(o[16 * hlf + 4 * v]) * inv_l,
                              __uint_as_float(o[16 * hlf + 4 * v + 1]) * inv_l,
                              __uint_as_float(o[16 * hlf + 4 * v + 2]) * inv_l,
                              __uint_as_float(o[16 * hlf + 4 * v + 3]) * inv_l);
            flush((int64_t)(32 * c + 16 * hlf) * 4);
          }
        } else {
          uint32_t wv[16];
          round_pack32<BF16>(o, inv_l, p.rounding, wv);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            *reinterpret_cast<uint4*>(stage + lane * 64 + ((v ^ (lane & 3)) * 16)) =
                make_uint4(wv[4 * v], wv[4 * v + 1], wv[4 * v + 2], wv[4 * v + 3]);
          flush((int64_t)(32 * c) * 2);
        }
      }
    }
    if (ok && row_ok && p.lse) {
      const int64_t li = p.dense ? ((int64_t)b * p.num_q_heads + head) * Sq + row0 + r
                                 : tok * p.num_q_heads + head;
      p.lse[li] = lse_v;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) report_status(p.status, kStatusTimeout);
}

template <bool BF16, bool FEAT>
cudaError_t launch_d256(const PrefillParams& p, dim3 grid, cudaStream_t stream) {
  static std::atomic<uint64_t> smem_set{0};
  const cudaError_t e = ensure_dynamic_smem(prefill_d256_kernel<BF16, FEAT>, kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  prefill_d256_kernel<BF16, FEAT><<<grid, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_d256(const PrefillParams& p, bool bf16, dim3 grid, cudaStream_t stream) {
  const bool feat = p.win_left >= 0 || p.win_right >= 0 || p.score_xform || p.sinks ||
                    p.out_scale != 1.f;
  if (feat) return bf16 ? launch_d256<true, true>(p, grid, stream) : launch_d256<false, true>(p, grid, stream);
  return bf16 ? launch_d256<true, false>(p, grid, stream) : launch_d256<false, false>(p, grid, stream);
}

}  // namespace attn

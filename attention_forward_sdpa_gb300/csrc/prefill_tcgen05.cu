// prefill_tcgen05.cu -- fused SDPA forward for prefill / dense attention on
// sm_103a: O = softmax(tau * Q K^T + mask) V by the online-softmax recurrence
// ("gfx942 unified attention, from the math up", sec. 3), over a paged K/V
// cache read through a block table (sec. 5), with the bottom-right causal mask
// and the early exit over fully-future key tiles (sec. 4), MHA and GQA.
//
// One CTA owns two 128-row query tiles that share one KV head: two heads of a
// GQA group over the same rows (balanced ping-pong), or, when the group size
// is odd, two consecutive row blocks of one head.  Warp roles:
//   warp 0      TMA producer (one thread): Q tiles once, then K_j / V_j tiles
//               (128 keys) into a ring of shared-memory slots (128-byte
//               swizzle), page by page through the block table;
//   warp 1      owns TMEM (512 columns); one thread issues the tcgen05 MMAs:
//               S_t = Q_t K_j^T (fp32 in TMEM), O_t += P_t V_j (P from TMEM);
//   warps 4-7   softmax for tile 0, warps 8-11 for tile 1 (one thread per
//               query row, tcgen05.ld of its row of S): mask, running max,
//               exp2, running denominator, P (16-bit) written back over S,
//               rescale of O in TMEM when the max moved, and the epilogue
//               O / l -> RTNE / RTNA / RTZ rounding -> global memory (a full
//               16-bit tile through shared memory and one TMA store, other
//               tiles through a per-warp staging buffer).
// The MMA issue order S_0(0), S_1(0), then per key tile PV_0(j), S_0(j+1),
// PV_1(j), S_1(j+1) lets one tile's softmax overlap the other tile's matrix
// products.  Every pipeline wait is bounded; one that runs out raises the
// CTA's abort flag and the status word records ATTN_ERR_TIMEOUT.
//
// The same kernel serves the dense strided entry point: then the page of a
// key tile is the batch index and Q / O are addressed by (batch, row, head)
// strides instead of packed rows.
//
// TMEM map (columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+d),
// O_1 [256+d, 256+2d).  P_t overwrites the first 64 columns of S_t as packed
// 16-bit pairs and is the A operand of the P.V product.

#include "attn_internal.h"
#include "round16.cuh"
#include "score_features.cuh"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;        // query rows per tile
constexpr int kBN = 128;        // keys per KV tile
constexpr int kThreads = 384;   // 12 warps
constexpr float kRescaleSlack = 8.f;  // log2 units: p stays <= 256

template <int D>
struct PrefillLayout {
  static constexpr int kHalves = D / 64;             // 128-byte swizzle spans 64 elements
  static constexpr int kHalfBytes = 128 * 128;       // 128 rows x 128 bytes
  static constexpr int kTileBytes = kHalves * kHalfBytes;
  static constexpr int kStages = D == 128 ? 4 : 8;   // K/V ring slots
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = 2 * kTileBytes;
  static constexpr int kBarOff = kRingOff + kStages * kTileBytes;
  static constexpr int kNumBars = 2 + 2 * kStages + 2 + 2 + 2 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // epilogue staging: 32 rows x 64 bytes per softmax warp (8 warps)
  // the sequence's first kPreIds page ids, loaded by the producer warp
  // during setup
  static constexpr int kPreIds = 128;
  static constexpr int kIdsOff = (kMiscOff + 16 + 15) / 16 * 16;
  static constexpr int kStageOff = (kIdsOff + kPreIds * 4 + 127) / 128 * 128;
  static constexpr int kSmemBytes = kStageOff + 8 * 2048 + 1024;  // + slack for 1024-byte alignment
  static __device__ __forceinline__ constexpr uint32_t s_col(int t) { return t ? 128u : 0u; }
  static __device__ __forceinline__ constexpr uint32_t o_col(int t) { return t ? 256u + D : 256u; }
  static constexpr uint32_t kTmemCols = 512;
};

// Waits without regard to the abort flag: used on the way out to make sure no
// asynchronous copy or MMA still targets this CTA's memory.
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
// sinks); without it the flags are compile-time off and the kernel carries
// none of their registers.
template <int D, bool BF16, bool FEAT>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
  using L = PrefillLayout<D>;
  const int win_left = FEAT ? p.win_left : -1;
  const int win_right = FEAT ? p.win_right : -1;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base + L::kQOff;
  const uint32_t sRing = base + L::kRingOff;
  const uint32_t bars = base + L::kBarOff;
  const uint32_t bar_q_full = bars;                                  // [2]
  const uint32_t bar_kv_full = bars + 8u * 2u;                       // [kStages]
  const uint32_t bar_kv_empty = bars + 8u * (2u + L::kStages);       // [kStages]
  const uint32_t bar_s_full = bars + 8u * (2u + 2u * L::kStages);    // [2]
  const uint32_t bar_p_full = bar_s_full + 16u;                      // [2]
  const uint32_t bar_o_full = bar_s_full + 32u;                      // [2]
  const uint32_t bar_mma_done = bar_s_full + 48u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ------------------------------------------------------------ work item
  const int b = blockIdx.y;
  int q_begin = 0, Sq = p.dense_sq, Sk = p.dense_sk;   // dense: rows are relative to the batch entry
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
  int head[2], row0[2], rows[2], n_kv[2], lim_lo[2];
  if (p.pair_heads) {
    if ((int)blockIdx.z >= n_rb) return;
    const int rb = n_rb - 1 - (int)blockIdx.z;   // heaviest (last) row block first
    for (int t = 0; t < 2; ++t) {
      head[t] = 2 * (int)blockIdx.x + t;
      row0[t] = rb * kBM;
    }
  } else {
    const int units = (n_rb + 1) / 2;
    if ((int)blockIdx.z >= units) return;
    const int u = units - 1 - (int)blockIdx.z;
    for (int t = 0; t < 2; ++t) {
      head[t] = (int)blockIdx.x;
      row0[t] = (2 * u + t) * kBM;
    }
  }
  const int off = Sk - Sq;  // bottom-right alignment: row i sees keys j <= i + off
  // Per tile: keys [lo, lim) of its rows (a sliding window narrows both
  // ends), the first key tile any row needs (jb), the end tile (n_kv), the
  // smallest upper limit (lim_lo) and the largest lower limit (lo_hi) -- the
  // tiles past lim_lo or before lo_hi need the per-element mask.
  int jb[2], lo_hi[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    rows[t] = row0[t] < Sq ? min(kBM, Sq - row0[t]) : 0;
    n_kv[t] = 0;
    lim_lo[t] = 0;
    jb[t] = 0;
    lo_hi[t] = 0;
    if (rows[t] > 0) {
      const int last = row0[t] + rows[t] - 1;
      int lim = Sk, first_lim = Sk;
      if (p.causal) {
        lim = min(lim, last + off + 1);
        first_lim = min(first_lim, row0[t] + off + 1);
      }
      if (win_right >= 0) {
        lim = min_sum(lim, last + off + 1, win_right);
        first_lim = min_sum(first_lim, row0[t] + off + 1, win_right);
      }
      int lo_first = 0;
      if (win_left >= 0) {
        lo_first = max(0, row0[t] + off - win_left);
        lo_hi[t] = max(0, last + off - win_left);
      }
      n_kv[t] = lim > lo_first ? (lim + kBN - 1) / kBN : 0;
      jb[t] = lo_first / kBN;
      lim_lo[t] = first_lim;
    }
  }
  // Both tiles walk the key tiles [j0, n_kv[t]) with j0 the earlier start:
  // the later-starting tile (a higher row block) sees its first tiles fully
  // masked.  cnt[t] = key tiles of tile t, counted from j0.
  const int j0 = !FEAT ? 0 : n_kv[0] > 0 ? (n_kv[1] > 0 ? min(jb[0], jb[1]) : jb[0]) : (n_kv[1] > 0 ? jb[1] : 0);
  int cnt[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) cnt[t] = n_kv[t] > 0 ? n_kv[t] - j0 : 0;
  const int n_kv_max = max(cnt[0], cnt[1]);
  // ALiBi raises the scores of the keys nearest the diagonal, so walked in
  // key order the running max climbs on every tile of a steep head and O is
  // rescaled each time.  With slopes, a CTA whose two tiles share one key
  // range (two heads of a KV head over the same rows) walks its key tiles
  // from the last to the first: the first tile then sets the max, and the
  // recurrence, exact in any order, rarely rescales.  key_tile(w) is the key
  // tile of walk step w.
  const bool rev = FEAT && p.alibi != nullptr && p.pair_heads;
  auto key_tile = [&](int w) -> int { return rev ? j0 + n_kv_max - 1 - w : j0 + w; };
  const int group = p.num_q_heads / p.num_kv_heads;
  const int kvh = head[0] / group;

  // ------------------------------------------------------------ setup
  // The producer warp fetches the sequence's first page ids now, so that the
  // first K/V copies do not wait for a dependent read of the block table
  // after setup; the loads overlap the barrier setup and TMEM allocation.
  int32_t* pre_ids = reinterpret_cast<int32_t*>(smem + L::kIdsOff);
  const int n_pre = p.dense ? 0 : min(L::kPreIds, (Sk + p.block_size - 1) / p.block_size);
  int32_t pre[L::kPreIds / 32];
  if (warp == 0) {
    const int32_t* btp = p.block_table + (int64_t)b * p.bt_stride;
#pragma unroll
    for (int k = 0; k < L::kPreIds / 32; ++k) {
      const int i = lane + 32 * k;
      pre[k] = i < n_pre ? btp[i] : 0;
    }
  }
  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_q_full + 8u * t, 1);
      mbar_init(bar_s_full + 8u * t, 1);
      mbar_init(bar_p_full + 8u * t, kBM);
      mbar_init(bar_o_full + 8u * t, 1);
    }
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar_kv_full + 8u * s, 1);
      mbar_init(bar_kv_empty + 8u * s, 1);
    }
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
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < L::kPreIds / 32; ++k) pre_ids[lane + 32 * k] = pre[k];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // page id `i` of the sequence: from shared memory when it was fetched above
  auto page_id = [&](const int32_t* btp, int i) -> int { return i < n_pre ? pre_ids[i] : btp[i]; };

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    // (stall_producer: a test of the timeout path issues no copy at all, so
    // that the first consumer wait runs out with nothing in flight)
    if (lane == 0 && !p.stall_producer) {
      for (int t = 0; t < 2; ++t) {
        if (n_kv[t] == 0) continue;
        const uint32_t bar = bar_q_full + 8u * t;
        mbar_arrive_expect_tx(bar, L::kTileBytes);
        for (int h = 0; h < L::kHalves; ++h) {
          const uint32_t dst = sQ + t * L::kTileBytes + h * L::kHalfBytes;
          if (p.dense) tma_load_4d(dst, &p.tm_q, bar, h * 64, head[t], row0[t], b);
          else tma_load_3d(dst, &p.tm_q, bar, h * 64, head[t], q_begin + row0[t]);
        }
      }
      const int bs = p.block_size;
      const int n_pages = (Sk + bs - 1) / bs;
      const int32_t* bt = p.block_table + (int64_t)b * p.bt_stride;
      int filled[L::kStages];
#pragma unroll
      for (int s = 0; s < L::kStages; ++s) filled[s] = 0;
      for (int i = 0; i < 2 * n_kv_max; ++i) {
        const int j = key_tile(i >> 1);
        const int s = i % L::kStages;
        const int u = i / L::kStages;
        if (u > 0 && !mbar_wait(bar_kv_empty + 8u * s, (u - 1) & 1, abort_flag, p.wait_limit_ns)) break;
        const uint32_t dst = sRing + s * L::kTileBytes;
        const uint32_t bar = bar_kv_full + 8u * s;
        const CUtensorMap* tm = (i & 1) ? &p.tm_v : &p.tm_k;
        const int key0 = j * kBN;
        if (bs >= kBN) {
          const int page = p.dense ? b : page_id(bt, key0 / bs);
          if (page < 0 || page >= p.num_blocks) report_status(p.status, kStatusBadBlockTable);
          mbar_arrive_expect_tx(bar, L::kTileBytes);
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_4d(dst + h * L::kHalfBytes, tm, bar, h * 64, kvh, key0 % bs, page);
        } else {
          const int first = key0 / bs;
          const int cnt = min(kBN / bs, n_pages - first);
          mbar_arrive_expect_tx(bar, (uint32_t)(cnt * L::kHalves * bs * 128));
          for (int r = 0; r < cnt; ++r) {
            const int page = page_id(bt, first + r);
            if (page < 0 || page >= p.num_blocks) report_status(p.status, kStatusBadBlockTable);
            for (int h = 0; h < L::kHalves; ++h)
              tma_load_4d(dst + h * L::kHalfBytes + r * bs * 128, tm, bar, h * 64, kvh, 0, page);
          }
        }
        filled[s] = u + 1;
      }
      // make sure no copy into this CTA's shared memory is still in flight
      for (int s = 0; s < L::kStages; ++s)
        if (filled[s] > 0) drain_wait(bar_kv_full + 8u * s, (filled[s] - 1) & 1, p.wait_limit_ns);
      for (int t = 0; t < 2; ++t)
        if (n_kv[t] > 0) drain_wait(bar_q_full + 8u * t, 0, p.wait_limit_ns);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------- MMA issuer
    // One thread: an MMA issue blocks for about one MMA's duration, so
    // every other instruction on this thread is tensor-pipe idle time.  The
    // shared-memory descriptors are built once; a K-step or a ring slot is
    // a constant added to the 16-byte address field (addresses < 256 KB).
    const uint32_t idesc_s = make_idesc_f16(BF16, kBM, kBN, false);
    const uint32_t idesc_pv = make_idesc_f16(BF16, kBM, D, true);
    const uint64_t dq0 = make_sdesc_sw128(sQ, 16, 1024);                  // Q_0, K-major
    const uint64_t dk0 = make_sdesc_sw128(sRing, 16, 1024);               // K in slot 0, K-major
    const uint64_t dv0 = make_sdesc_sw128(sRing, L::kHalfBytes, 1024);    // V in slot 0, MN-major
    constexpr uint64_t kTileStep = L::kTileBytes >> 4;
    auto issue_s = [&](int t, int slot) {
      const uint64_t a = dq0 + (uint64_t)t * kTileStep;
      const uint64_t b = dk0 + (uint64_t)slot * kTileStep;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t o = (uint64_t)(((kk >> 2) * L::kHalfBytes + (kk & 3) * 32) >> 4);
        umma_ss(tmem + L::s_col(t), a + o, b + o, idesc_s, kk > 0 ? 1u : 0u);
      }
    };
    auto issue_pv = [&](int t, int slot, bool acc) {
      const uint64_t b = dv0 + (uint64_t)slot * kTileStep;
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk)
        umma_ts(tmem + L::o_col(t), tmem + L::s_col(t) + kk * 8, b + (uint64_t)((kk * 16 * 128) >> 4),
                idesc_pv, (acc || kk > 0) ? 1u : 0u);
    };
    const int nk0 = cnt[0], nk1 = cnt[1];
    bool ok = true;
    if (nk0 > 0) ok = mbar_wait(bar_q_full, 0, abort_flag, p.wait_limit_ns);
    if (ok && nk1 > 0) ok = mbar_wait(bar_q_full + 8u, 0, abort_flag, p.wait_limit_ns);
    if (ok && n_kv_max > 0) {
      ok = mbar_wait(bar_kv_full, 0, abort_flag, p.wait_limit_ns);  // K_0: slot 0, first fill
      if (ok) {
        tc_fence_after();
        if (nk0 > 0) {
          issue_s(0, 0);
          umma_commit(bar_s_full);
        }
        if (nk1 > 0) {
          issue_s(1, 0);
          umma_commit(bar_s_full + 8u);
        }
        umma_commit(bar_kv_empty);
      }
    }
    // per key tile j: PV_0(j), S_0(j+1), PV_1(j), S_1(j+1)
    for (int j = 0; ok && j < n_kv_max; ++j) {
      const int iv = 2 * j + 1;                    // V_j
      const int sv = iv % L::kStages;
      if (!mbar_wait(bar_kv_full + 8u * sv, (iv / L::kStages) & 1, abort_flag, p.wait_limit_ns)) break;
      tc_fence_after();
      const int jk = key_tile(j);
      if ((jk + 1) * kBN > Sk) {
        // keys at or past kv_len in the last tile: their V rows may hold
        // anything (NaN included); P is 0 there but 0 * NaN is not, so zero them.
        const int r0 = Sk - jk * kBN;
        uint8_t* vt = smem + (sRing - base) + sv * L::kTileBytes;
        for (int idx = 0; idx < (kBN - r0) * L::kHalves * 8; ++idx) {
          const int chunk = idx & 7;
          const int rh = idx >> 3;
          const int h = rh % L::kHalves;
          const int r = r0 + rh / L::kHalves;
          *reinterpret_cast<uint4*>(vt + h * L::kHalfBytes + r * 128 + chunk * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      const int ik = iv + 1;                       // K_{j+1}
      const int sk = ik % L::kStages;
      const bool s0 = j + 1 < nk0, s1 = j + 1 < nk1;
      if (j < nk0) {
        if (!mbar_wait(bar_p_full, j & 1, abort_flag, p.wait_limit_ns)) break;
        tc_fence_after();
        issue_pv(0, sv, j > 0);
      }
      if (s0 || s1) {
        if (!mbar_wait(bar_kv_full + 8u * sk, (ik / L::kStages) & 1, abort_flag, p.wait_limit_ns)) break;
        tc_fence_after();
      }
      if (j < nk0) {
        if (s0) {
          issue_s(0, sk);
          umma_commit(bar_s_full);
        } else {
          umma_commit(bar_o_full);
        }
      }
      if (j < nk1) {
        if (!mbar_wait(bar_p_full + 8u, j & 1, abort_flag, p.wait_limit_ns)) break;
        tc_fence_after();
        issue_pv(1, sv, j > 0);
        if (s1) {
          issue_s(1, sk);
          umma_commit(bar_s_full + 8u);
        } else {
          umma_commit(bar_o_full + 8u);
        }
      }
      umma_commit(bar_kv_empty + 8u * sv);
      if (s0 || s1) umma_commit(bar_kv_empty + 8u * sk);
    }
    // no MMA may still be running when TMEM is released
    umma_commit(bar_mma_done);
    drain_wait(bar_mma_done, 0, p.wait_limit_ns);
  } else if (warp >= 4) {
    // ---------------------------------------------------------- softmax + epilogue
    const int t = (warp - 4) >> 2;
    const int wq = warp & 3;
    // this tile's bounds as scalars (a runtime index into the arrays would
    // put them in local memory)
    const int t_row0 = t ? row0[1] : row0[0];
    const int t_rows = t ? rows[1] : rows[0];
    const int t_nkv = t ? cnt[1] : cnt[0];
    const int t_limlo = t ? lim_lo[1] : lim_lo[0];
    const int t_lohi = t ? lo_hi[1] : lo_hi[0];
    const int t_head = t ? head[1] : head[0];
    const int r = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + L::s_col(t);
    const uint32_t tO = tmem + lane_off + L::o_col(t);
    const int i_row = t_row0 + r;
    int key_lim = p.causal ? min(Sk, i_row + off + 1) : Sk;
    if (win_right >= 0) key_lim = min_sum(key_lim, i_row + off + 1, win_right);
    const int key_lo = win_left >= 0 ? i_row + off - win_left : 0;
    const float sl2 = p.scale_log2;
    const float slope = FEAT && p.alibi ? p.alibi[t_head] : 0.f;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int jr = 0; jr < t_nkv; ++jr) {
      const int j = key_tile(jr);            // key tile
      if (!mbar_wait(bar_s_full + 8u * t, jr & 1, abort_flag, p.wait_limit_ns)) { ok = false; break; }
      tc_fence_after();
      uint32_t s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, s[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait(s[c]);
      if (FEAT && p.score_xform) rewrite_scores(s, p.scale, p.softcap, slope, (float)(i_row + off - j * kBN));
      if ((j + 1) * kBN > t_limlo || (FEAT && j * kBN < t_lohi)) {
        const int cl = key_lim - j * kBN;  // columns >= cl are masked for this row
        const int cf = key_lo - j * kBN;   // and columns < cf
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (32 * c + e >= cl || (FEAT && 32 * c + e < cf)) s[c][e] = 0xFF800000u;  // -inf
      }
      // row max over the tile's 128 scores: four independent chains of
      // three-input maxima (one per 32-column chunk), then one merge
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
      // The running max is only raised when the tile's max exceeds it by
      // more than kRescaleSlack (log2 units).  Any reference value works for
      // the recurrence as long as o and l use the same one, so this is exact;
      // it keeps p <= 2^kRescaleSlack and makes the O rescale rare.
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
      if (jr > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
        // O_t is final for tile j-1 here: S_t(j) was issued after PV_t(j-1)
        // and its commit covers every earlier MMA.
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
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
      mbar_arrive(bar_p_full + 8u * t);
      const float2 r01 = fadd2(rs[0], rs[1]), r23 = fadd2(rs[2], rs[3]);
      l = l * alpha + ((r01.x + r23.x) + (r01.y + r23.y));
      m = m_new;
    }
    if (ok && t_nkv > 0) {
      ok = mbar_wait(bar_o_full + 8u * t, 0, abort_flag, p.wait_limit_ns);
      tc_fence_after();
    }
    const bool row_ok = r < t_rows;
    const int64_t tok = (int64_t)q_begin + t_row0 + r;
    float inv_l, lse_v;
    finish_row(m, l, FEAT && p.sinks ? p.sinks[t_head] : -INFINITY, inv_l, lse_v);
    if (FEAT) inv_l *= p.out_scale;   // fp8 V factor (1 otherwise)
    if (t_rows == kBM && p.rounding != 3) {
      // Full tile, 16-bit output: the rows are written into this tile's Q
      // slot (free: the o_full commit covers every product that read it) in
      // the 128-byte-swizzled layout of the Q map, and one thread stores the
      // tile with TMA.  All 128 threads reach the barrier, whatever ok says.
      if (ok) {
        uint8_t* qt = smem + L::kQOff + t * L::kTileBytes;
        // two 32-column chunks per TMEM round trip
#pragma unroll
        for (int c2 = 0; c2 < D / 64; ++c2) {
          uint32_t o[2][32];
          if (t_nkv > 0) {
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
            // columns [64 c2 + 32 hc, +32): half c2, 16-byte chunks 4 hc .. 4 hc + 3
            uint8_t* rowp = qt + c2 * L::kHalfBytes + r * 128;
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
      named_bar_sync(1 + t, kBM);
      if (wq == 0 && lane == 0 && ok && *abort_flag == 0) {
#pragma unroll
        for (int h = 0; h < L::kHalves; ++h) {
          const uint32_t src = sQ + t * L::kTileBytes + h * L::kHalfBytes;
          if (p.dense) tma_store_4d(&p.tm_o, src, h * 64, t_head, t_row0, b);
          else tma_store_3d(&p.tm_o, src, h * 64, t_head, q_begin + t_row0);
        }
        bulk_commit_group();
        bulk_wait_group_read0();
      }
    } else if (ok) {
      // The warp writes its 32 rows through a 2 KB staging buffer so that
      // each store instruction covers 8 rows x 64 contiguous bytes instead of
      // 32 rows x 16 bytes.  Row i of the buffer holds 64 bytes of row i, its
      // four 16-byte pieces rotated by (i & 3) to spread the banks.
      uint8_t* stage = smem + L::kStageOff + (warp - 4) * 2048;
      // element offset of this warp's first row and the distance between rows
      const int64_t row_elems = p.dense ? p.o_stride_s : (int64_t)p.num_q_heads * D;
      const int64_t tile_base =
          p.dense ? (int64_t)b * p.o_stride_b + (int64_t)(t_row0 + wq * 32) * p.o_stride_s +
                        (int64_t)t_head * p.o_stride_h
                  : ((int64_t)q_begin + t_row0 + wq * 32) * row_elems + (int64_t)t_head * D;
      const int rows_here = min(32, t_rows - wq * 32);   // valid rows of this warp
      auto flush = [&](int64_t col_byte) {                // write 64 bytes per row
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
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (t_nkv > 0) {
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
      // packed: [total_q, Hq]; dense: [batch, Hq, Sq]
      const int64_t li = p.dense ? ((int64_t)b * p.num_q_heads + t_head) * Sq + t_row0 + r
                                 : tok * p.num_q_heads + t_head;
      p.lse[li] = lse_v;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) report_status(p.status, kStatusTimeout);
}

template <int D, bool BF16, bool FEAT>
cudaError_t launch_one_f(const PrefillParams& p, dim3 grid, cudaStream_t stream) {
  using L = PrefillLayout<D>;
  static std::atomic<uint64_t> smem_set{0};
  const cudaError_t e = ensure_dynamic_smem(prefill_kernel<D, BF16, FEAT>, L::kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  prefill_kernel<D, BF16, FEAT><<<grid, kThreads, L::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_one(const PrefillParams& p, dim3 grid, cudaStream_t stream) {
  const bool feat = p.win_left >= 0 || p.win_right >= 0 || p.score_xform || p.sinks ||
                    p.out_scale != 1.f;
  return feat ? launch_one_f<D, BF16, true>(p, grid, stream) : launch_one_f<D, BF16, false>(p, grid, stream);
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, int head_size, bool bf16, dim3 grid,
                           cudaStream_t stream) {
  if (head_size == 128) return bf16 ? launch_one<128, true>(p, grid, stream) : launch_one<128, false>(p, grid, stream);
  if (head_size == 64) return bf16 ? launch_one<64, true>(p, grid, stream) : launch_one<64, false>(p, grid, stream);
  if (head_size == 256) return launch_prefill_d256(p, bf16, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn

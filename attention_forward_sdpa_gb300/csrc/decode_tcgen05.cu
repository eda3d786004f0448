// decode_tcgen05.cu -- split-KV decode ("gfx942 unified attention, from the
// math up", sec. 8) for head size 128 as a persistent, TMA-fed, tcgen05
// kernel.  Decode is bound by HBM bandwidth (each K/V byte is read once and
// used for 2 * G flops), so the design goal is a continuous stream of page
// loads with almost no instructions per byte:
//
//   * work items are (sequence, group of query heads sharing a KV head,
//     split); persistent CTAs (one per SM) claim them from an atomic counter,
//     so items of different length balance dynamically and the load pipeline
//     never drains between items;
//   * warp 0 streams each item's Q rows and its pages as 16-row TMA boxes
//     (128-byte swizzle) into a ring of 32 KB key tiles (K and V alternate);
//     its lanes issue the boxes of a tile in parallel;
//   * warp 1 issues S^T = K Q^T (M = 128 keys, N = 16 query heads, fp32 in
//     TMEM) and O^T += V^T P^T (M = 128 channels, N = 16): with the keys on M
//     one thread owns one key's scores;
//   * warps 2-5 (one thread per key, then per channel) take each tile's
//     scores from TMEM, form the running max across the CTA, exp2, the
//     running denominators, write P^T (16-bit) to shared memory, rescale O^T
//     in TMEM when the max moved, and at the end of an item write the partial
//     state (un-normalised o, max in log2 units, denominator) -- or, with one
//     split, the final rounded output.
// S^T is double-buffered so the next tile's product overlaps this tile's
// softmax.  Every wait is bounded (see sm103_ptx.cuh); the CTA-wide exchange
// of the softmax warps also goes through an mbarrier so that it is bounded.

#include "attn_internal.h"
#include "round16.cuh"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kD = 128;                 // head size handled here
constexpr int kTK = 128;                // keys per tile
constexpr int kThreads = 192;
constexpr int kSlots = 6;               // K/V ring slots of one tile each
constexpr int kItemRing = 4;
constexpr int kTileBytes = kTK * kD * 2;        // 32 KB
constexpr int kHalfBytes = kTK * 128;           // 128 keys x 64 channels
constexpr int kQBytes = 2 * 16 * 128;           // two channel halves of [16 heads][64]
constexpr int kPBytes = 2 * 16 * 128;           // two key halves of [16 heads][64 keys]
constexpr float kLn2 = 0.693147180559945309f;

struct ItemEntry {
  int b;       // sequence, or -1 at the end of the work
  int hg;      // head group: query heads [hg * heads_per_item, ...)
  int split;
  int k0, k1;  // key range
  int pad[3];
};

constexpr int kRingOff = 0;
constexpr int kQOff = kRingOff + kSlots * kTileBytes;
constexpr int kPOff = kQOff + 2 * kQBytes;
constexpr int kRedOff = kPOff + 2 * kPBytes;            // float [2][4][16]
constexpr int kLRedOff = kRedOff + 2 * 4 * 16 * 4;      // float [2][4][16]
constexpr int kItemOff = kLRedOff + 2 * 4 * 16 * 4;     // ItemEntry [kItemRing]
constexpr int kBarOff = kItemOff + kItemRing * (int)sizeof(ItemEntry);
// barriers: kv_full[kSlots] kv_empty[kSlots] q_full[2] q_empty[2] s_full[2]
//           p_full[2] pv_done item_full[R] item_empty[R] mma_done red
constexpr int kNumBars = 2 * kSlots + 2 + 2 + 2 + 2 + 1 + 2 * kItemRing + 1 + 1;
constexpr int kMiscOff = kBarOff + kNumBars * 8;
constexpr int kSmemBytes = kMiscOff + 16 + 1024;
constexpr uint32_t kTmemCols = 64;      // S^T x 2 (16 columns each), O^T (16)
constexpr uint32_t kOCol = 32u;

__device__ __forceinline__ uint32_t s_col(uint32_t g) { return (g & 1u) ? 16u : 0u; }

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) break;
  }
}

// Keys of split s of a sequence of length Sk: [s*per, min(Sk, (s+1)*per)) with
// per = ceil(ceil(Sk / splits) / 16) * 16 (the same rule as the SIMT path).
__device__ __forceinline__ void split_keys(int Sk, int splits, int s, int& k0, int& k1) {
  int per = (Sk + splits - 1) / splits;
  per = (per + 15) / 16 * 16;
  k0 = min(Sk, s * per);
  k1 = min(Sk, k0 + per);
}

// Byte offset of the 16-bit P^T element (head h, key k) in the K-major,
// 128-byte-swizzled B operand: two key halves of [16 heads][64 keys].
__device__ __forceinline__ uint32_t p_offset(int h, int k) {
  const int half = k >> 6, c = k & 63;
  const int chunk = (c >> 3) ^ (h & 7);
  return (uint32_t)(half * 2048 + h * 128 + chunk * 16 + (c & 7) * 2);
}

template <bool BF16, int NH>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sRing = base + kRingOff;
  const uint32_t sQ = base + kQOff;
  const uint32_t sP = base + kPOff;
  float* red = reinterpret_cast<float*>(smem + kRedOff);
  float* lred = reinterpret_cast<float*>(smem + kLRedOff);
  ItemEntry* items = reinterpret_cast<ItemEntry*>(smem + kItemOff);
  const uint32_t bars = base + kBarOff;
  const uint32_t bar_kv_full = bars;
  const uint32_t bar_kv_empty = bars + 8u * kSlots;
  const uint32_t bar_q_full = bars + 8u * (2 * kSlots);
  const uint32_t bar_q_empty = bar_q_full + 16u;
  const uint32_t bar_s_full = bar_q_full + 32u;
  const uint32_t bar_p_full = bar_q_full + 48u;
  const uint32_t bar_pv_done = bar_q_full + 64u;
  const uint32_t bar_item_full = bar_pv_done + 8u;
  const uint32_t bar_item_empty = bar_item_full + 8u * kItemRing;
  const uint32_t bar_mma_done = bar_item_empty + 8u * kItemRing;
  const uint32_t bar_red = bar_mma_done + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int GH = p.heads_per_item;
  const int hgroups = p.num_q_heads / GH;
  const int G = p.num_q_heads / p.num_kv_heads;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar_kv_full + 8u * s, 1);
      mbar_init(bar_kv_empty + 8u * s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_q_full + 8u * i, 1);
      mbar_init(bar_q_empty + 8u * i, 1);
      mbar_init(bar_s_full + 8u * i, 1);
      mbar_init(bar_p_full + 8u * i, 128);
    }
    mbar_init(bar_pv_done, 1);
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(bar_item_full + 8u * i, 1);
      mbar_init(bar_item_empty + 8u * i, 1 + 4);
    }
    mbar_init(bar_mma_done, 1);
    mbar_init(bar_red, 128);
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
    const int bs = p.block_size;
    uint32_t seen = 0, q_loads = 0, fills = 0;
    uint32_t last_fill[kSlots];
#pragma unroll
    for (int s = 0; s < kSlots; ++s) last_fill[s] = 0;
    for (;;) {
      int item = 0;
      if (lane == 0) item = atomicAdd(p.counter, 1);
      item = __shfl_sync(0xFFFFFFFFu, item, 0);
      const bool end = item >= p.n_items;
      int b = -1, hg = 0, split = 0, k0 = 0, k1 = 0;
      if (!end) {
        split = item % p.num_splits;
        const int rest = item / p.num_splits;
        hg = rest % hgroups;
        b = rest / hgroups;
        int Sk = p.seq_lens[b];
        if (Sk < 0 || Sk > p.max_seqlen_k) {
          if (lane == 0) report_status(p.status, kStatusBadArg);
          Sk = 0;
        }
        split_keys(Sk, p.num_splits, split, k0, k1);
      }
      const uint32_t rs = seen % kItemRing;
      if (seen >= kItemRing &&
          !mbar_wait(bar_item_empty + 8u * rs, ((seen / kItemRing) - 1) & 1, abort_flag))
        break;
      if (lane == 0) {
        ItemEntry e;
        e.b = b; e.hg = hg; e.split = split; e.k0 = k0; e.k1 = k1;
        e.pad[0] = e.pad[1] = e.pad[2] = 0;
        items[rs] = e;
        mbar_arrive(bar_item_full + 8u * rs);
      }
      __syncwarp();
      ++seen;
      if (end) break;
      const int n_tiles = (k1 - k0 + kTK - 1) / kTK;
      if (n_tiles == 0) continue;
      const int kvh = (hg * GH) / G;
      // Q rows of the head group
      const uint32_t qs = q_loads & 1u;
      if (q_loads >= 2 && !mbar_wait(bar_q_empty + 8u * qs, ((q_loads >> 1) - 1) & 1, abort_flag))
        break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_q_full + 8u * qs, (uint32_t)(2 * p.q_box_rows * 128));
        for (int h = 0; h < 2; ++h)
          tma_load_3d(sQ + qs * kQBytes + h * 2048, &p.tm_q, bar_q_full + 8u * qs, h * 64, hg * GH, b);
      }
      ++q_loads;
      const int32_t* bt = p.block_table + (int64_t)b * p.bt_stride;
      bool ok = true;
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int tk0 = k0 + t * kTK;
        const int nbox = (min(kTK, k1 - tk0) + 15) / 16;
        int page = 0, row = 0;
        if (lane < nbox) {
          const int key = tk0 + 16 * lane;
          page = bt[key / bs];
          row = key % bs;
          if (page < 0 || page >= p.num_blocks) report_status(p.status, kStatusBadBlockTable);
        }
        for (int kind = 0; kind < 2; ++kind) {
          const uint32_t s = fills % kSlots;
          if (fills >= kSlots &&
              !mbar_wait(bar_kv_empty + 8u * s, ((fills / kSlots) - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t bar = bar_kv_full + 8u * s;
          if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(nbox * 2 * 2048));
          __syncwarp();
          if (lane < nbox) {
            const CUtensorMap* tm = kind ? &p.tm_v : &p.tm_k;
            const uint32_t dst = sRing + s * kTileBytes + lane * 16 * 128;
            tma_load_4d(dst, tm, bar, 0, kvh, row, page);
            tma_load_4d(dst + kHalfBytes, tm, bar, 64, kvh, row, page);
          }
          last_fill[s] = fills + 1;
          ++fills;
        }
      }
      if (!ok) break;
    }
    // no copy may still be in flight into this CTA's shared memory
    if (lane == 0) {
      for (int s = 0; s < kSlots; ++s)
        if (last_fill[s] > 0) drain_wait(bar_kv_full + 8u * s, (last_fill[s] - 1) / kSlots & 1);
      for (uint32_t i = (q_loads > 2 ? q_loads - 2 : 0); i < q_loads; ++i)
        drain_wait(bar_q_full + 8u * (i & 1u), (i >> 1) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    const bool leader = lane == 0;
    const uint32_t idesc_s = make_idesc_f16(BF16, 128, 16, false, false);
    const uint32_t idesc_pv = make_idesc_f16(BF16, 128, 16, false, true);
    uint32_t seen = 0, q_uses = 0, fills = 0, g = 0;
    bool have_pending = false, ok = true;
    uint32_t pend_g = 0, pend_fill = 0;
    bool pend_first = false;
    auto flush_pv = [&]() -> bool {
      if (!mbar_wait(bar_p_full + 8u * (pend_g & 1u), (pend_g >> 1) & 1, abort_flag)) return false;
      const uint32_t sv = pend_fill % kSlots;
      if (!mbar_wait(bar_kv_full + 8u * sv, (pend_fill / kSlots) & 1, abort_flag)) return false;
      tc_fence_after();
      if (leader) {
        const uint32_t a0 = sRing + sv * kTileBytes;
        const uint32_t b0 = sP + (pend_g & 1u) * kPBytes;
#pragma unroll
        for (int kk = 0; kk < kTK / 16; ++kk) {
          umma_ss(tmem + kOCol, make_sdesc_sw128(a0 + kk * 16 * 128, kHalfBytes, 1024),
                  make_sdesc_sw128(b0 + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024), idesc_pv,
                  (pend_first && kk == 0) ? 0u : 1u);
        }
        umma_commit(bar_pv_done);
        umma_commit(bar_kv_empty + 8u * sv);
      }
      __syncwarp();
      return true;
    };
    for (;;) {
      const uint32_t rs = seen % kItemRing;
      if (!mbar_wait(bar_item_full + 8u * rs, (seen / kItemRing) & 1, abort_flag)) { ok = false; break; }
      const ItemEntry e = items[rs];
      __syncwarp();
      if (leader) mbar_arrive(bar_item_empty + 8u * rs);
      ++seen;
      if (e.b < 0) break;
      const int n_tiles = (e.k1 - e.k0 + kTK - 1) / kTK;
      if (n_tiles == 0) continue;
      const uint32_t qs = q_uses & 1u;
      if (!mbar_wait(bar_q_full + 8u * qs, (q_uses >> 1) & 1, abort_flag)) { ok = false; break; }
      ++q_uses;
      for (int t = 0; t < n_tiles && ok; ++t) {
        const uint32_t sk = fills % kSlots;
        if (!mbar_wait(bar_kv_full + 8u * sk, (fills / kSlots) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        if (leader) {
          const uint32_t a0 = sRing + sk * kTileBytes;
          const uint32_t b0 = sQ + qs * kQBytes;
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t oa = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
            const uint32_t ob = (kk >> 2) * 2048 + (kk & 3) * 32;
            umma_ss(tmem + s_col(g), make_sdesc_sw128(a0 + oa, 16, 1024),
                    make_sdesc_sw128(b0 + ob, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(bar_s_full + 8u * (g & 1u));
          umma_commit(bar_kv_empty + 8u * sk);
          if (t == n_tiles - 1) umma_commit(bar_q_empty + 8u * qs);
        }
        __syncwarp();
        ++fills;
        if (have_pending && !flush_pv()) { ok = false; break; }
        have_pending = true;
        pend_g = g;
        pend_fill = fills;   // V of this tile is the next fill
        pend_first = t == 0;
        ++fills;
        ++g;
      }
      if (!ok) break;
      // finish the item now so that its epilogue does not wait for the next
      // item's first key tile
      if (!flush_pv()) { ok = false; break; }
      have_pending = false;
    }
    if (ok && have_pending) flush_pv();
    if (leader) umma_commit(bar_mma_done);
    __syncwarp();
    drain_wait(bar_mma_done, 0);
  } else {
    // ---------------------------------------------------------- softmax + epilogue
    const int sw = warp - 2;                 // 0..3
    const int quarter = warp & 3;            // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;       // key (for S^T) / channel (for O^T)
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    const int Hq = p.num_q_heads;
    uint32_t seen = 0, g = 0, red_uses = 0;
    bool ok = true;
    auto cta_sync = [&]() -> bool {  // the 128 softmax threads
      mbar_arrive(bar_red);
      const bool r_ok = mbar_wait(bar_red, red_uses & 1u, abort_flag);
      ++red_uses;
      return r_ok;
    };
    for (;;) {
      const uint32_t rs = seen % kItemRing;
      if (!mbar_wait(bar_item_full + 8u * rs, (seen / kItemRing) & 1, abort_flag)) { ok = false; break; }
      const ItemEntry e = items[rs];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_item_empty + 8u * rs);
      ++seen;
      if (e.b < 0) break;
      const int n_tiles = (e.k1 - e.k0 + kTK - 1) / kTK;
      float m[NH], lp[NH];
#pragma unroll
      for (int h = 0; h < NH; ++h) { m[h] = -INFINITY; lp[h] = 0.f; }
      for (int t = 0; t < n_tiles && ok; ++t) {
        if (!mbar_wait(bar_s_full + 8u * (g & 1u), (g >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[NH];
        tmem_ld_n<NH>(tmem + lane_off + s_col(g), sv);
        tmem_ld_wait_n<NH>(sv);
        const int key = e.k0 + t * kTK + r;
        const bool valid = key < e.k1;
        float x[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) x[h] = valid ? __uint_as_float(sv[h]) * sl2 : -INFINITY;
        // CTA-wide max per head
        float* rb = red + (red_uses & 1u) * 64;
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          float v = x[h];
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
          if (lane == 0) rb[sw * 16 + h] = v;
        }
        if (!cta_sync()) { ok = false; break; }
        float alpha[NH], mu[NH];
        bool rescale = false;
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          const float tm = fmaxf(fmaxf(rb[h], rb[16 + h]), fmaxf(rb[32 + h], rb[48 + h]));
          const float mn = fmaxf(m[h], tm);
          mu[h] = mn == -INFINITY ? 0.f : mn;
          alpha[h] = fast_exp2(m[h] - mu[h]);
          rescale |= alpha[h] != 1.f;
          m[h] = mn;
        }
        float pr[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          pr[h] = fast_exp2(x[h] - mu[h]);
          lp[h] = fmaf(lp[h], alpha[h], pr[h]);
        }
        // PV of the previous tile must be complete before O^T and the P^T
        // buffer of two tiles ago are touched
        if (g >= 1) {
          if (!mbar_wait(bar_pv_done, (g - 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
        }
        if (t > 0 && rescale) {
          uint32_t ov[NH];
          tmem_ld_n<NH>(tmem + lane_off + kOCol, ov);
          tmem_ld_wait_n<NH>(ov);
#pragma unroll
          for (int h = 0; h < NH; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha[h]);
          tmem_st_n<NH>(tmem + lane_off + kOCol, ov);
          tmem_st_wait();
        }
        if (!valid) {
          // this key's V row may hold another split's key, a stale tile or
          // poison: P is 0 there, but 0 * NaN is not, so zero the row
          const uint32_t fill_v = 2u * g + 1u;
          const uint32_t sv_slot = fill_v % kSlots;
          if (!mbar_wait(bar_kv_full + 8u * sv_slot, (fill_v / kSlots) & 1, abort_flag)) { ok = false; break; }
          uint8_t* vrow = smem + (sRing - base) + sv_slot * kTileBytes + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(vrow + kHalfBytes + c * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        uint8_t* pb = smem + (sP - base) + (g & 1u) * kPBytes;
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          const uint16_t v = BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(pr[h]))
                                  : __half_as_ushort(__float2half_rn(pr[h]));
          *reinterpret_cast<uint16_t*>(pb + p_offset(h, r)) = v;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar_p_full + 8u * (g & 1u));
        ++g;
      }
      if (!ok) break;
      // ---- item epilogue: denominators, then partial or final output
      float o[NH];
      if (n_tiles > 0) {
        if (!mbar_wait(bar_pv_done, (g - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        uint32_t ov[NH];
        tmem_ld_n<NH>(tmem + lane_off + kOCol, ov);
        tmem_ld_wait_n<NH>(ov);
#pragma unroll
        for (int h = 0; h < NH; ++h) o[h] = __uint_as_float(ov[h]);
      } else {
#pragma unroll
        for (int h = 0; h < NH; ++h) o[h] = 0.f;
      }
      float* lb = lred + (red_uses & 1u) * 64;
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        float v = lp[h];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        if (lane == 0) lb[sw * 16 + h] = v;
      }
      if (!cta_sync()) { ok = false; break; }
      const int h0 = e.hg * GH;
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        if (h >= GH) break;
        const float L = (lb[h] + lb[16 + h]) + (lb[32 + h] + lb[48 + h]);
        const int64_t row = (int64_t)e.b * Hq + h0 + h;
        if (p.num_splits > 1) {
          p.part_o[(row * p.num_splits + e.split) * kD + r] = o[h];
          if (r == 0) {
            p.part_ml[(row * p.num_splits + e.split) * 2 + 0] = m[h];
            p.part_ml[(row * p.num_splits + e.split) * 2 + 1] = L;
          }
        } else {
          const float v = L > 0.f ? o[h] / L : 0.f;
          if (p.rounding == 3) static_cast<float*>(p.out)[row * kD + r] = v;
          else static_cast<uint16_t*>(p.out)[row * kD + r] = round_out<BF16>(v, p.rounding);
          if (r == 0 && p.lse) p.lse[row] = L > 0.f ? m[h] * kLn2 + logf(L) : -INFINITY;
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) report_status(p.status, kStatusTimeout);
}

template <bool BF16, int NH>
cudaError_t launch_t(const DecodeParams& p, int grid, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<BF16, NH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  decode_tc_kernel<BF16, NH><<<grid, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

// Splits of one decode step on the tcgen05 path (head size 128, heads per
// item <= 16).  The caller has zeroed p.counter on `stream`.
cudaError_t launch_decode_tc(const DecodeParams& p, bool bf16, int grid, cudaStream_t stream) {
  const int gh = p.heads_per_item;
  if (gh <= 4) return bf16 ? launch_t<true, 4>(p, grid, stream) : launch_t<false, 4>(p, grid, stream);
  if (gh <= 8) return bf16 ? launch_t<true, 8>(p, grid, stream) : launch_t<false, 8>(p, grid, stream);
  return bf16 ? launch_t<true, 16>(p, grid, stream) : launch_t<false, 16>(p, grid, stream);
}

}  // namespace attn

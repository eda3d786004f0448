// prefill_streamk.cu -- the prefill of prefill_tcgen05.cu as a persistent
// kernel with a stream-K schedule, so that no SM idles behind a fractional
// last wave or waits for the heaviest causal row blocks alone.
//
// Work units are the ones of the one-shot kernel: two 128-row query tiles
// that share a KV head (two heads of a GQA group over the same rows, or two
// consecutive row blocks of one head), each with its own number of key tiles
// (causal rows see fewer).  All key tiles of all units, laid end to end
// (sequence, head unit, row unit, key tile), form one sequence of T tiles;
// CTA c of the G persistent CTAs takes tiles [c T / G, (c + 1) T / G).  A
// range cuts at most two units, so every CTA has the same work up to one key
// tile.  This is the tail split for the fractional last wave of [MM] "Dónde
// viven los datos y por qué 16x16x16" taken to its limit: every split point
// is placed where the load balances, not only in the last wave.
//
// A unit cut across CTAs is merged by the CTA that finishes its part last:
// every part stores its un-normalised o, running max m (log2 units) and
// denominator l for the unit's rows in a workspace slot of its own, then
// counts itself on the unit's ticket; the part that completes the count
// reads every part back and merges them in key order -- M = max m_s,
// O = sum 2^(m_s - M) o_s / sum 2^(m_s - M) l_s, the log-sum-exp combine of
// "gfx942 unified attention, from the math up", sec. 8 -- so the result does
// not depend on which part finished last.  Tickets carry the call's epoch:
// a ticket left by an earlier call (or never written) reads as empty, so the
// workspace needs no clearing between calls.
//
// Warp roles as in the one-shot kernel: warp 0 computes the segments of its
// range and publishes them to a small ring in shared memory, then streams Q
// and K/V tiles with TMA; warp 1 issues the tcgen05 MMAs; warps 4-7 / 8-11
// run the softmax of query tile 0 / 1 and the epilogue.  Output rows go out
// through per-warp staging buffers, so that a Q slot can take the next
// segment's tile as soon as the last S = Q K^T product of a segment has read
// it.  Every wait is bounded.

#include "attn_internal.h"
#include "round16.cuh"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;        // query rows per tile
constexpr int kBN = 128;        // keys per KV tile
constexpr int kThreads = 384;   // 12 warps
constexpr float kRescaleSlack = 8.f;
constexpr int kSegRing = 4;
constexpr float kLn2 = 0.693147180559945309f;

// One segment of a CTA's range: key tiles [ja, jb) of one unit.
struct Seg {
  int b;          // sequence; -1 ends the work
  int q_begin, Sq, Sk;
  int x, z;       // head unit, row unit
  int ja, jb;     // key tiles of the unit this segment covers
  int n_unit;     // key tiles of the whole unit
  int c_first;    // CTA whose range holds the unit's first key tile: the ticket
  int n_segs;     // parts the unit is cut into (1: this segment is the whole unit)
  int slot;       // workspace slot of this part
};

template <int D>
struct SkLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalfBytes = 128 * 128;
  static constexpr int kTileBytes = kHalves * kHalfBytes;
  static constexpr int kStages = D == 128 ? 4 : 8;
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = 2 * kTileBytes;
  static constexpr int kBarOff = kRingOff + kStages * kTileBytes;
  // q_full[2] q_empty[2] kv_full[S] kv_empty[S] s_full[2] p_full[2] o_full[2]
  // seg_full[R] seg_empty[R] pub tk mma_done
  static constexpr int kNumBars = 2 + 2 + 2 * kStages + 2 + 2 + 2 + 2 * kSegRing + 3;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;              // tmem slot, abort, last flag
  static constexpr int kSegOff = (kMiscOff + 16 + 15) / 16 * 16;
  // per-sequence tables: int64 tile prefix and zero-unit prefix [kSkMaxSeqs + 1],
  // int32 q_begin, Sq, Sk, zero units per head unit [kSkMaxSeqs]
  static constexpr int kSeqOff = (kSegOff + kSegRing * (int)sizeof(Seg) + 7) / 8 * 8;
  static constexpr int kZeroOff = kSeqOff + (kSkMaxSeqs + 1) * 8;
  static constexpr int kQbOff = kZeroOff + (kSkMaxSeqs + 1) * 8;
  static constexpr int kSqOff = kQbOff + kSkMaxSeqs * 4;
  static constexpr int kSkOff = kSqOff + kSkMaxSeqs * 4;
  static constexpr int kZuOff = kSkOff + kSkMaxSeqs * 4;
  static constexpr int kStageOff = (kZuOff + kSkMaxSeqs * 4 + 127) / 128 * 128;
  static constexpr int kSmemBytes = kStageOff + 8 * 2048 + 1024;
  static __device__ __forceinline__ constexpr uint32_t s_col(int t) { return t ? 128u : 0u; }
  static __device__ __forceinline__ constexpr uint32_t o_col(int t) { return t ? 256u + D : 256u; }
  static constexpr uint32_t kTmemCols = 512;
};

__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long atom_cas_acq_rel_gpu_u64(unsigned long long* p,
                                                                     unsigned long long cmp,
                                                                     unsigned long long val) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.cas.b64 %0, [%1], %2, %3;"
               : "=l"(old)
               : "l"(p), "l"(cmp), "l"(val)
               : "memory");
  return old;
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) break;
  }
}

// Key tiles a query row block needs: rows up to `last` see keys j <= last + off
// (causal, bottom-right aligned) or all Sk keys.
__device__ __forceinline__ int key_tiles(int last, int off, int Sk, bool causal) {
  int lim = Sk;
  if (causal) lim = min(lim, last + off + 1);
  return lim > 0 ? (lim + kBN - 1) / kBN : 0;
}

// Key tiles of row unit z of a sequence (the larger count of its two tiles).
__device__ __forceinline__ int unit_tiles(int z, int Sq, int Sk, bool pair, bool causal) {
  const int rows = pair ? kBM : 2 * kBM;
  const int last = min(z * rows + rows - 1, Sq - 1);
  return key_tiles(last, Sk - Sq, Sk, causal);
}

// CTA whose range [c T / G, (c + 1) T / G) holds key tile `pos`.
__device__ __forceinline__ int cta_of(int64_t pos, int64_t T, int G) {
  int c = (int)(pos * G / T);
  while (c + 1 < G && (int64_t)(c + 1) * T / G <= pos) ++c;
  while (c > 0 && (int64_t)c * T / G > pos) --c;
  return c;
}

// One row of the output: D fp32 values (64 at a time from `get`, as two
// 32-column chunks) times inv_l, rounded, written by the warp through its
// 2 KB staging buffer (each store instruction covers 8 rows x 64 contiguous
// bytes).  Every lane calls this (warp-uniform); rows >= rows_here are not
// stored.
template <int D, bool BF16, typename Get>
__device__ __forceinline__ void store_rows(const PrefillParams& p, uint8_t* stage, int lane,
                                           int64_t tile_base, int64_t row_elems, int rows_here,
                                           float inv_l, Get get) {
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
  auto put = [&](const uint32_t (&o)[32], int c) {
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
  };
#pragma unroll 1
  for (int c2 = 0; c2 < D / 64; ++c2) {
    uint32_t o[2][32];
    get(c2, o[0], o[1]);
    put(o[0], 2 * c2);
    put(o[1], 2 * c2 + 1);
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1) prefill_sk_kernel(const __grid_constant__ PrefillParams p) {
  using L = SkLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base + L::kQOff;
  const uint32_t sRing = base + L::kRingOff;
  const uint32_t bars = base + L::kBarOff;
  const uint32_t bar_q_full = bars;                                   // [2]
  const uint32_t bar_q_empty = bars + 16u;                            // [2]
  const uint32_t bar_kv_full = bars + 32u;                            // [kStages]
  const uint32_t bar_kv_empty = bar_kv_full + 8u * L::kStages;        // [kStages]
  const uint32_t bar_s_full = bar_kv_empty + 8u * L::kStages;         // [2]
  const uint32_t bar_p_full = bar_s_full + 16u;                       // [2]
  const uint32_t bar_o_full = bar_s_full + 32u;                       // [2]
  const uint32_t bar_seg_full = bar_s_full + 48u;                     // [kSegRing]
  const uint32_t bar_seg_empty = bar_seg_full + 8u * kSegRing;        // [kSegRing]
  const uint32_t bar_pub = bar_seg_empty + 8u * kSegRing;
  const uint32_t bar_tk = bar_pub + 8u;
  const uint32_t bar_mma_done = bar_tk + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 8);
  Seg* segs = reinterpret_cast<Seg*>(smem + L::kSegOff);
  int64_t* seq_start = reinterpret_cast<int64_t*>(smem + L::kSeqOff);   // key tiles before sequence b
  int64_t* zero_start = reinterpret_cast<int64_t*>(smem + L::kZeroOff); // zero-tile units before b
  int* t_qb = reinterpret_cast<int*>(smem + L::kQbOff);
  int* t_sq = reinterpret_cast<int*>(smem + L::kSqOff);
  int* t_sk = reinterpret_cast<int*>(smem + L::kSkOff);
  int* t_zu = reinterpret_cast<int*>(smem + L::kZuOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool pair = p.pair_heads != 0;
  const bool causal = p.causal != 0;
  const int G = (int)gridDim.x;
  const int cta = (int)blockIdx.x;
  const int group = p.num_q_heads / p.num_kv_heads;

  // ------------------------------------------------------------ setup
  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_q_full + 8u * t, 1);
      mbar_init(bar_q_empty + 8u * t, 1);
      mbar_init(bar_s_full + 8u * t, 1);
      mbar_init(bar_p_full + 8u * t, kBM);
      mbar_init(bar_o_full + 8u * t, 1);
    }
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar_kv_full + 8u * s, 1);
      mbar_init(bar_kv_empty + 8u * s, 1);
    }
    for (int s = 0; s < kSegRing; ++s) {
      mbar_init(bar_seg_full + 8u * s, 1);
      mbar_init(bar_seg_empty + 8u * s, 1 + 8);   // the MMA thread and the 8 softmax warps
    }
    mbar_init(bar_pub, 8);                         // the 8 softmax warps
    mbar_init(bar_tk, 1);
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- schedule
    // The warp builds the per-sequence tables, a lane per sequence: key
    // tiles of all its units (a malformed sequence counts as empty and is
    // reported) and its zero-tile units -- rows that see no key at all
    // (causal rows above a diagonal offset below zero, or Sk = 0), which get
    // only their zero output.  Lane 0 then walks the CTA's range.
    const int nseq = p.num_seqs;
    const int units_rows = pair ? kBM : 2 * kBM;
    const int ux = p.sk_units_x;
    int64_t carry = 0, zcarry = 0;
    if (lane == 0) {
      seq_start[0] = 0;
      zero_start[0] = 0;
    }
    for (int b0 = 0; b0 < nseq; b0 += 32) {
      const int b = b0 + lane;
      int64_t tiles = 0;
      int zu = 0;
      if (b < nseq) {
        int q0 = 0, Sq = p.dense_sq, Sk = p.dense_sk;
        if (!p.dense) {
          q0 = p.query_start_loc[b];
          const int q1 = p.query_start_loc[b + 1];
          Sq = q1 - q0;
          Sk = p.seq_lens[b];
          if (q0 < 0 || Sq < 0 || Sq > p.max_seqlen_q || q1 > p.total_q || Sk < 0 || Sk > p.max_seqlen_k) {
            report_status(p.status, kStatusBadArg);
            Sq = 0;
          }
        }
        const int n_ru = (Sq + units_rows - 1) / units_rows;
        if (causal) {
          for (int z = 0; z < n_ru; ++z) {
            const int n = unit_tiles(z, Sq, Sk, pair, causal);
            tiles += n;
            zu += n == 0;
          }
        } else {
          const int n = Sk > 0 ? (Sk + kBN - 1) / kBN : 0;
          tiles = (int64_t)n * n_ru;
          zu = n == 0 ? n_ru : 0;
        }
        t_qb[b] = q0;
        t_sq[b] = Sq;
        t_sk[b] = Sk;
        t_zu[b] = zu;
      }
      int64_t v = tiles * ux, w = (int64_t)zu * ux;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t vn = __shfl_up_sync(0xFFFFFFFFu, v, o);
        const int64_t wn = __shfl_up_sync(0xFFFFFFFFu, w, o);
        if (lane >= o) {
          v += vn;
          w += wn;
        }
      }
      if (b < nseq) {
        seq_start[b + 1] = carry + v;
        zero_start[b + 1] = zcarry + w;
      }
      carry += __shfl_sync(0xFFFFFFFFu, v, 31);
      zcarry += __shfl_sync(0xFFFFFFFFu, w, 31);
    }
    __syncwarp();
    const int64_t T = carry;        // key tiles of all units
    const int64_t Zn = zcarry;      // zero-tile units
    // CTAs 0 .. Ge-1 share the T tiles (Ge <= T: no range is empty)
    const int Ge = (int)(T < (int64_t)G ? T : (int64_t)G);

    if (lane == 0) {
      // ---------------------------------------------------------- producer
      int64_t pos = cta < Ge ? (int64_t)cta * T / Ge : 0;
      const int64_t end = cta < Ge ? (int64_t)(cta + 1) * T / Ge : 0;
      int b = 0, q0 = 0, Sq = 0, Sk = 0, x = 0, z = 0, ja = 0;
      auto load_seq = [&](int bb) {
        q0 = t_qb[bb];
        Sq = t_sq[bb];
        Sk = t_sk[bb];
      };
      if (pos < end) {
        while (b + 1 < nseq && seq_start[b + 1] <= pos) ++b;
        load_seq(b);
        const int64_t per_x = (seq_start[b + 1] - seq_start[b]) / ux;
        int64_t r = pos - seq_start[b];
        x = (int)(r / per_x);
        r -= (int64_t)x * per_x;
        for (;;) {
          const int n = unit_tiles(z, Sq, Sk, pair, causal);
          if (r < n) break;
          r -= n;
          ++z;
        }
        ja = (int)r;
      }
      // zero-tile units e = cta, cta + G, ... (usually none)
      int64_t ze = cta;
      int zb = 0;
      uint32_t sidx = 0, fill = 0;
      int qn[2] = {0, 0};
      bool ok = true;
      for (;;) {
        const bool zero_unit = ze < Zn;
        const bool done = !zero_unit && !(pos < end);
        const uint32_t rs = sidx % kSegRing;
        if (sidx >= kSegRing &&
            !mbar_wait(bar_seg_empty + 8u * rs, ((sidx / kSegRing) - 1) & 1, abort_flag, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        Seg sg;
        sg.b = -1;
        int n_unit = 0, jb = 0;
        if (zero_unit) {
          while (zb + 1 < nseq && zero_start[zb + 1] <= ze) ++zb;
          const int64_t r = ze - zero_start[zb];
          sg.b = zb;
          sg.q_begin = t_qb[zb];
          sg.Sq = t_sq[zb];
          sg.Sk = t_sk[zb];
          sg.x = (int)(r / t_zu[zb]);
          sg.z = (int)(r % t_zu[zb]);
          sg.ja = sg.jb = sg.n_unit = 0;
          sg.c_first = cta;
          sg.n_segs = 1;
          sg.slot = -1;
          segs[rs] = sg;
          mbar_arrive(bar_seg_full + 8u * rs);
          ++sidx;
          ze += G;
          continue;
        }
        if (!done) {
          n_unit = unit_tiles(z, Sq, Sk, pair, causal);
          const int64_t take = min((int64_t)(n_unit - ja), end - pos);
          jb = ja + (int)take;
          sg.b = b;
          sg.q_begin = q0;
          sg.Sq = Sq;
          sg.Sk = Sk;
          sg.x = x;
          sg.z = z;
          sg.ja = ja;
          sg.jb = jb;
          sg.n_unit = n_unit;
          if (ja == 0 && jb == n_unit) {
            sg.c_first = cta;
            sg.n_segs = 1;
            sg.slot = -1;
          } else {
            const int64_t first = pos - ja;
            sg.c_first = cta_of(first, T, Ge);
            sg.n_segs = cta_of(first + n_unit - 1, T, Ge) - sg.c_first + 1;
            sg.slot = cta == sg.c_first ? 2 * cta + 1 : 2 * cta;   // tail part / head part of a range
          }
        }
        segs[rs] = sg;
        mbar_arrive(bar_seg_full + 8u * rs);   // release: the entry is visible to whoever waits
        ++sidx;
        if (done) break;
        // Q tiles of the segment's unit (a tile with no key tile here is skipped)
        int head[2], row0[2], cnt[2];
        for (int t = 0; t < 2; ++t) {
          head[t] = pair ? 2 * x + t : x;
          row0[t] = pair ? z * kBM : (2 * z + t) * kBM;
          const int rows = row0[t] < Sq ? min(kBM, Sq - row0[t]) : 0;
          const int nk = rows > 0 ? key_tiles(row0[t] + rows - 1, Sk - Sq, Sk, causal) : 0;
          cnt[t] = max(0, min(jb, nk) - ja);
        }
        for (int t = 0; t < 2 && ok; ++t) {
          if (cnt[t] == 0) continue;
          if (qn[t] > 0 && !mbar_wait(bar_q_empty + 8u * t, (qn[t] - 1) & 1, abort_flag, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          const uint32_t bar = bar_q_full + 8u * t;
          mbar_arrive_expect_tx(bar, L::kTileBytes);
          for (int h = 0; h < L::kHalves; ++h) {
            const uint32_t dst = sQ + t * L::kTileBytes + h * L::kHalfBytes;
            if (p.dense) tma_load_4d(dst, &p.tm_q, bar, h * 64, head[t], row0[t], b);
            else tma_load_3d(dst, &p.tm_q, bar, h * 64, head[t], q0 + row0[t]);
          }
          ++qn[t];
        }
        if (!ok) break;
        // K / V tiles ja .. ja + n_max - 1
        const int n_max = max(cnt[0], cnt[1]);
        const int kvh = head[0] / group;
        const int bs = p.block_size;
        const int n_pages = (Sk + bs - 1) / bs;
        const int32_t* bt = p.block_table + (int64_t)b * p.bt_stride;
        for (int i = 0; i < 2 * n_max; ++i, ++fill) {
          const int j = ja + (i >> 1);
          const uint32_t s = fill % L::kStages;
          const uint32_t u = fill / L::kStages;
          if (u > 0 && !mbar_wait(bar_kv_empty + 8u * s, (u - 1) & 1, abort_flag, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          const uint32_t dst = sRing + s * L::kTileBytes;
          const uint32_t bar = bar_kv_full + 8u * s;
          const CUtensorMap* tm = (i & 1) ? &p.tm_v : &p.tm_k;
          const int key0 = j * kBN;
          if (bs >= kBN) {
            const int page = p.dense ? b : bt[key0 / bs];
            if (page < 0 || page >= p.num_blocks) report_status(p.status, kStatusBadBlockTable);
            mbar_arrive_expect_tx(bar, L::kTileBytes);
            for (int h = 0; h < L::kHalves; ++h)
              tma_load_4d(dst + h * L::kHalfBytes, tm, bar, h * 64, kvh, key0 % bs, page);
          } else {
            const int first = key0 / bs;
            const int cp = min(kBN / bs, n_pages - first);
            mbar_arrive_expect_tx(bar, (uint32_t)(cp * L::kHalves * bs * 128));
            for (int r = 0; r < cp; ++r) {
              const int page = bt[first + r];
              if (page < 0 || page >= p.num_blocks) report_status(p.status, kStatusBadBlockTable);
              for (int h = 0; h < L::kHalves; ++h)
                tma_load_4d(dst + h * L::kHalfBytes + r * bs * 128, tm, bar, h * 64, kvh, 0, page);
            }
          }
        }
        if (!ok) break;
        // advance to the next unit when this one is finished
        pos += jb - ja;
        ja = jb;
        if (ja == n_unit && pos < end) {
          ja = 0;
          const int n_ru = (Sq + units_rows - 1) / units_rows;
          if (++z >= n_ru) {
            z = 0;
            if (++x >= p.sk_units_x) {
              x = 0;
              // next sequence with work
              do { ++b; } while (b + 1 < nseq && seq_start[b + 1] == seq_start[b]);
              load_seq(b);
            }
          }
        }
      }
      // no copy may still target this CTA's memory on the way out
      for (uint32_t k = (fill > (uint32_t)L::kStages ? fill - L::kStages : 0); k < fill; ++k)
        drain_wait(bar_kv_full + 8u * (k % L::kStages), (k / L::kStages) & 1, p.wait_limit_ns);
      for (int t = 0; t < 2; ++t)
        if (qn[t] > 0) drain_wait(bar_q_full + 8u * t, (qn[t] - 1) & 1, p.wait_limit_ns);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------- MMA issuer
    const uint32_t idesc_s = make_idesc_f16(BF16, kBM, kBN, false);
    const uint32_t idesc_pv = make_idesc_f16(BF16, kBM, D, true);
    const uint64_t dq0 = make_sdesc_sw128(sQ, 16, 1024);
    const uint64_t dk0 = make_sdesc_sw128(sRing, 16, 1024);
    const uint64_t dv0 = make_sdesc_sw128(sRing, L::kHalfBytes, 1024);
    constexpr uint64_t kTileStep = L::kTileBytes >> 4;
    auto issue_s = [&](int t, int slot) {
      const uint64_t a = dq0 + (uint64_t)t * kTileStep;
      const uint64_t bdesc = dk0 + (uint64_t)slot * kTileStep;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t o = (uint64_t)(((kk >> 2) * L::kHalfBytes + (kk & 3) * 32) >> 4);
        umma_ss(tmem + L::s_col(t), a + o, bdesc + o, idesc_s, kk > 0 ? 1u : 0u);
      }
    };
    auto issue_pv = [&](int t, int slot, bool acc) {
      const uint64_t bdesc = dv0 + (uint64_t)slot * kTileStep;
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk)
        umma_ts(tmem + L::o_col(t), tmem + L::s_col(t) + kk * 8, bdesc + (uint64_t)((kk * 16 * 128) >> 4),
                idesc_pv, (acc || kk > 0) ? 1u : 0u);
    };
    uint32_t sidx = 0, fc = 0;
    int qc[2] = {0, 0}, pc[2] = {0, 0};
    bool ok = true;
    for (;;) {
      const uint32_t rs = sidx % kSegRing;
      if (!mbar_wait(bar_seg_full + 8u * rs, (sidx / kSegRing) & 1, abort_flag, p.wait_limit_ns)) break;
      const Seg sg = segs[rs];
      mbar_arrive(bar_seg_empty + 8u * rs);
      ++sidx;
      if (sg.b < 0) break;
      int cnt[2];
      for (int t = 0; t < 2; ++t) {
        const int row0 = pair ? sg.z * kBM : (2 * sg.z + t) * kBM;
        const int rows = row0 < sg.Sq ? min(kBM, sg.Sq - row0) : 0;
        const int nk = rows > 0 ? key_tiles(row0 + rows - 1, sg.Sk - sg.Sq, sg.Sk, causal) : 0;
        cnt[t] = max(0, min(sg.jb, nk) - sg.ja);
      }
      const int nk0 = cnt[0], nk1 = cnt[1];
      const int n_max = max(nk0, nk1);
      if (n_max == 0) continue;               // a zero-tile unit: nothing to multiply
      if (nk0 > 0) ok = mbar_wait(bar_q_full, qc[0] & 1, abort_flag, p.wait_limit_ns);
      if (ok && nk1 > 0) ok = mbar_wait(bar_q_full + 8u, qc[1] & 1, abort_flag, p.wait_limit_ns);
      if (!ok) break;
      if (nk0 > 0) ++qc[0];
      if (nk1 > 0) ++qc[1];
      // K of the first key tile, then S_0, S_1
      {
        const uint32_t s = fc % L::kStages;
        if (!mbar_wait(bar_kv_full + 8u * s, (fc / L::kStages) & 1, abort_flag, p.wait_limit_ns)) break;
        tc_fence_after();
        for (int t = 0; t < 2; ++t) {
          if ((t ? nk1 : nk0) == 0) continue;
          issue_s(t, (int)s);
          umma_commit(bar_s_full + 8u * t);
        }
        umma_commit(bar_kv_empty + 8u * s);
      }
      for (int j = 0; ok && j < n_max; ++j) {
        const uint32_t iv = fc + 2u * j + 1u;     // V_j
        const uint32_t sv = iv % L::kStages;
        if (!mbar_wait(bar_kv_full + 8u * sv, (iv / L::kStages) & 1, abort_flag, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int jk = sg.ja + j;                  // key tile of the unit
        if ((jk + 1) * kBN > sg.Sk) {
          // keys at or past kv_len: their V rows may hold anything; P is 0
          // there but 0 * NaN is not, so zero them
          const int r0 = sg.Sk - jk * kBN;
          uint8_t* vt = smem + (sRing - base) + sv * L::kTileBytes;
          for (int idx = 0; idx < (kBN - r0) * L::kHalves * 8; ++idx) {
            const int chunk = idx & 7;
            const int rh = idx >> 3;
            const int h = rh % L::kHalves;
            const int r = r0 + rh / L::kHalves;
            *reinterpret_cast<uint4*>(vt + h * L::kHalfBytes + r * 128 + chunk * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        const uint32_t ik = iv + 1u;               // K_{j+1}
        const uint32_t sk = ik % L::kStages;
        const bool s0 = j + 1 < nk0, s1 = j + 1 < nk1;
        if (j < nk0) {
          if (!mbar_wait(bar_p_full, pc[0] & 1, abort_flag, p.wait_limit_ns)) { ok = false; break; }
          ++pc[0];
          tc_fence_after();
          issue_pv(0, (int)sv, j > 0);
        }
        if (s0 || s1) {
          if (!mbar_wait(bar_kv_full + 8u * sk, (ik / L::kStages) & 1, abort_flag, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        if (j < nk0) {
          if (s0) {
            issue_s(0, (int)sk);
            umma_commit(bar_s_full);
          } else {
            umma_commit(bar_o_full);
          }
        }
        if (j < nk1) {
          if (!mbar_wait(bar_p_full + 8u, pc[1] & 1, abort_flag, p.wait_limit_ns)) { ok = false; break; }
          ++pc[1];
          tc_fence_after();
          issue_pv(1, (int)sv, j > 0);
          if (s1) {
            issue_s(1, (int)sk);
            umma_commit(bar_s_full + 8u);
          } else {
            umma_commit(bar_o_full + 8u);
          }
        }
        umma_commit(bar_kv_empty + 8u * sv);
        if (s0 || s1) umma_commit(bar_kv_empty + 8u * sk);
      }
      if (!ok) break;
      fc += 2u * (uint32_t)n_max;
    }
    umma_commit(bar_mma_done);
    drain_wait(bar_mma_done, 0, p.wait_limit_ns);
  } else if (warp >= 4) {
    // ---------------------------------------------------------- softmax + epilogue
    const int t = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + L::s_col(t);
    const uint32_t tO = tmem + lane_off + L::o_col(t);
    uint8_t* stage = smem + L::kStageOff + (warp - 4) * 2048;
    const float sl2 = p.scale_log2;
    uint32_t sidx = 0;
    int sph = 0, oph = 0, npub = 0;
    bool ok = true;
    for (;;) {
      const uint32_t rs = sidx % kSegRing;
      if (!mbar_wait(bar_seg_full + 8u * rs, (sidx / kSegRing) & 1, abort_flag, p.wait_limit_ns)) break;
      __syncwarp();
      const Seg sg = segs[rs];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_seg_empty + 8u * rs);
      __syncwarp();                          // converged before the TMEM accesses that follow
      ++sidx;
      if (sg.b < 0) break;
      const int head = pair ? 2 * sg.x + t : sg.x;
      const int row0 = pair ? sg.z * kBM : (2 * sg.z + t) * kBM;
      const int rows = row0 < sg.Sq ? min(kBM, sg.Sq - row0) : 0;
      const int off = sg.Sk - sg.Sq;
      const int nk = rows > 0 ? key_tiles(row0 + rows - 1, off, sg.Sk, causal) : 0;
      const int cnt = max(0, min(sg.jb, nk) - sg.ja);
      const int lim_lo = causal ? min(sg.Sk, row0 + off + 1) : sg.Sk;   // smallest row limit of the tile
      const int i_row = row0 + r;
      const int key_lim = causal ? min(sg.Sk, i_row + off + 1) : sg.Sk;
      float m = -INFINITY, l = 0.f;
      for (int jr = 0; jr < cnt; ++jr) {
        const int j = sg.ja + jr;
        if (!mbar_wait(bar_s_full + 8u * t, sph & 1, abort_flag, p.wait_limit_ns)) { ok = false; break; }
        ++sph;
        tc_fence_after();
        uint32_t s[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, s[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_wait(s[c]);
        if ((j + 1) * kBN > lim_lo) {
          const int cl = key_lim - j * kBN;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (32 * c + e >= cl) s[c][e] = 0xFF800000u;
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
        // lazy running max (exact: any reference works if o and l share it)
        const float mxs = mx * sl2;
        const float m_new = (mxs > m + kRescaleSlack) ? mxs : m;
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = fast_exp2(m - m_use);
        const float2 sc2 = make_float2(sl2, sl2);
        const float2 nm2 = make_float2(-m_use, -m_use);
        float2 rsum[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) rsum[a] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 xx = ffma2(make_float2(__uint_as_float(s[c][2 * e]), __uint_as_float(s[c][2 * e + 1])),
                                    sc2, nm2);
            const float2 pp = make_float2(fast_exp2(xx.x), fast_exp2(xx.y));
            rsum[e & 3] = fadd2(rsum[e & 3], pp);
            pk[e] = BF16 ? pack_bf16x2_rn(pp.x, pp.y) : pack_f16x2_rn(pp.x, pp.y);
          }
          tmem_st16(tS + 16 * c, pk);
        }
        if (jr > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
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
        const float2 r01 = fadd2(rsum[0], rsum[1]), r23 = fadd2(rsum[2], rsum[3]);
        l = l * alpha + ((r01.x + r23.x) + (r01.y + r23.y));
        m = m_new;
      }
      if (!ok) break;
      if (cnt > 0) {
        if (!mbar_wait(bar_o_full + 8u * t, oph & 1, abort_flag, p.wait_limit_ns)) break;
        ++oph;
        tc_fence_after();
      }
      const int rows_here = min(32, rows - wq * 32);   // rows of this warp inside the tile
      const int64_t row_elems = p.dense ? p.o_stride_s : (int64_t)p.num_q_heads * D;
      const int64_t tile_base =
          p.dense ? (int64_t)sg.b * p.o_stride_b + (int64_t)(row0 + wq * 32) * p.o_stride_s +
                        (int64_t)head * p.o_stride_h
                  : ((int64_t)sg.q_begin + row0 + wq * 32) * row_elems + (int64_t)head * D;
      const bool row_ok = r < rows;
      // A full tile with 16-bit output leaves through this tile's Q slot
      // (free: o_full covers every product that read it) and one TMA store;
      // the slot goes back to the producer (q_empty) once the store has read
      // it.  Other tiles go through the staging buffers and hand the slot
      // back at once.  Every thread of the tile calls this.
      const bool tma_out = rows == kBM && p.rounding != 3;
      auto write_tile = [&](float inv_l, auto get) {
        if (tma_out) {
          uint8_t* qt = smem + L::kQOff + t * L::kTileBytes;
#pragma unroll 1
          for (int c2 = 0; c2 < D / 64; ++c2) {
            uint32_t o[2][32];
            get(c2, o[0], o[1]);
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
              uint32_t w[16];
              round_pack32<BF16>(o[hc], inv_l, p.rounding, w);
              uint8_t* rowp = qt + c2 * L::kHalfBytes + r * 128;
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const int chunk = hc * 4 + v;
                *reinterpret_cast<uint4*>(rowp + ((chunk ^ (r & 7)) * 16)) =
                    make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
              }
            }
          }
          fence_proxy_async_smem();
          named_bar_sync(1 + t, kBM);
          if (wq == 0 && lane == 0) {
            for (int h = 0; h < L::kHalves; ++h) {
              const uint32_t src = sQ + t * L::kTileBytes + h * L::kHalfBytes;
              if (p.dense) tma_store_4d(&p.tm_o, src, h * 64, head, row0, sg.b);
              else tma_store_3d(&p.tm_o, src, h * 64, head, sg.q_begin + row0);
            }
            bulk_commit_group();
            bulk_wait_group_read0();
          }
        } else {
          store_rows<D, BF16>(p, stage, lane, tile_base, row_elems, rows_here, inv_l, get);
        }
        if (cnt > 0 && wq == 0 && lane == 0) mbar_arrive(bar_q_empty + 8u * t);
      };
      auto lse_index = [&]() -> int64_t {
        return p.dense ? ((int64_t)sg.b * p.num_q_heads + head) * sg.Sq + row0 + r
                       : ((int64_t)sg.q_begin + row0 + r) * p.num_q_heads + head;
      };
      if (sg.n_segs == 1) {
        // the whole unit: normalise and store
        float inv_l, lse_v;
        if (l != 0.f) {
          inv_l = 1.f / l;
          lse_v = m * kLn2 + logf(l);
        } else {
          inv_l = 0.f;
          lse_v = -INFINITY;
        }
        write_tile(inv_l, [&](int c2, uint32_t(&o0)[32], uint32_t(&o1)[32]) {
          if (cnt > 0) {
            tmem_ld32(tO + 64 * c2, o0);
            tmem_ld32(tO + 64 * c2 + 32, o1);
            tmem_ld_wait(o0);
            tmem_ld_wait(o1);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o0[e] = o1[e] = 0u;
          }
        });
        if (row_ok && p.lse) p.lse[lse_index()] = lse_v;
        continue;
      }
      // ---- part of a unit: publish (o, m, l) in this part's slot.  Layout
      // [slot][tile][D / 4][128 rows] of float4, so that a warp's 32 rows of
      // one 4-column group are 512 contiguous bytes (one coalesced access).
      const int64_t row_id = ((int64_t)sg.slot * 2 + t) * kBM + r;
      float4* po = reinterpret_cast<float4*>(p.sk_part_o) + ((int64_t)sg.slot * 2 + t) * (D / 4) * kBM + r;
#pragma unroll 1
      for (int c2 = 0; c2 < D / 64; ++c2) {
        uint32_t o[2][32];
        if (cnt > 0) {
          tmem_ld32(tO + 64 * c2, o[0]);
          tmem_ld32(tO + 64 * c2 + 32, o[1]);
          tmem_ld_wait(o[0]);
          tmem_ld_wait(o[1]);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[0][e] = o[1][e] = 0u;
        }
#pragma unroll
        for (int hc = 0; hc < 2; ++hc)
#pragma unroll
          for (int v = 0; v < 8; ++v)
            __stcg(po + (int64_t)(16 * c2 + 8 * hc + v) * kBM,
                   make_float4(__uint_as_float(o[hc][4 * v]), __uint_as_float(o[hc][4 * v + 1]),
                               __uint_as_float(o[hc][4 * v + 2]), __uint_as_float(o[hc][4 * v + 3])));
      }
      if (cnt > 0 && wq == 0 && lane == 0) mbar_arrive(bar_q_empty + 8u * t);   // the slot was not used
      __stcg(reinterpret_cast<float2*>(p.sk_part_ml) + row_id, make_float2(m, l));
      // both tiles published (the CTA barrier below orders every thread's
      // stores before the ticket thread's release), then one thread counts
      // this part on the ticket
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pub);
      const bool pub_ok = mbar_wait(bar_pub, npub & 1, abort_flag, p.wait_limit_ns);
      __syncwarp();
      if (!pub_ok) break;
      if (warp == 4 && lane == 0) {
        // release: this CTA's partial stores (ordered before this thread by
        // the barrier) become visible before the count; acquire: the parts
        // counted before it are visible to this CTA's merge reads
        unsigned long long* tk = p.sk_ticket + sg.c_first;
        const unsigned long long tag = p.sk_epoch & 0xFFFFFFFFFFFFull;
        unsigned long long cur = ld_relaxed_gpu_u64(tk);
        unsigned long long want;
        for (;;) {
          want = (cur >> 16) == tag ? cur + 1ull : ((tag << 16) | 1ull);
          const unsigned long long prev = atom_cas_acq_rel_gpu_u64(tk, cur, want);
          if (prev == cur) break;
          cur = prev;
        }
        *last_flag = (int)(want & 0xFFFFull) == sg.n_segs ? 1 : 0;
        mbar_arrive(bar_tk);
      }
      const bool tk_ok = mbar_wait(bar_tk, npub & 1, abort_flag, p.wait_limit_ns);
      __syncwarp();
      ++npub;
      if (!tk_ok) break;
      if (!*last_flag) continue;
      // ---- the last part: merge every part of the unit in key order.  The
      // thread's row: M = max m_s, then L = sum 2^(m_s - M) l_s, then o in
      // 64-column blocks, every part's 64 values loaded before they are used.
      const int n_s = sg.n_segs;
      auto slot_of = [&](int k) { return k == 0 ? 2 * sg.c_first + 1 : 2 * (sg.c_first + k); };
      auto row_of = [&](int k) { return ((int64_t)slot_of(k) * 2 + t) * kBM + r; };
      float M = -INFINITY;
      for (int k = 0; k < n_s; ++k) M = fmaxf(M, __ldcg(reinterpret_cast<const float2*>(p.sk_part_ml) + row_of(k)).x);
      const float Mu = M == -INFINITY ? 0.f : M;
      float Lm = 0.f;
      for (int k = 0; k < n_s; ++k) {
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.sk_part_ml) + row_of(k));
        Lm = fmaf(fast_exp2(ml.x - Mu), ml.y, Lm);
      }
      float inv_l, lse_v;
      if (Lm != 0.f) {
        inv_l = 1.f / Lm;
        lse_v = Mu * kLn2 + logf(Lm);
      } else {
        inv_l = 0.f;
        lse_v = -INFINITY;
      }
      store_rows<D, BF16>(p, stage, lane, tile_base, row_elems, rows_here, inv_l,
                          [&](int c2, uint32_t(&o0)[32], uint32_t(&o1)[32]) {
        // columns [64 c2, 64 c2 + 64): every part's block, 16 loads in flight
        float acc[64];
#pragma unroll
        for (int e = 0; e < 64; ++e) acc[e] = 0.f;
        for (int k = 0; k < n_s; ++k) {
          const int64_t rid = row_of(k);
          const float w = fast_exp2(__ldcg(reinterpret_cast<const float2*>(p.sk_part_ml) + rid).x - Mu);
          const float4* src = reinterpret_cast<const float4*>(p.sk_part_o) +
                              ((int64_t)slot_of(k) * 2 + t) * (D / 4) * kBM + r + (int64_t)(16 * c2) * kBM;
          float4 q4[16];
#pragma unroll
          for (int v = 0; v < 16; ++v) q4[v] = __ldcg(src + (int64_t)v * kBM);
#pragma unroll
          for (int v = 0; v < 16; ++v) {
            acc[4 * v] = fmaf(w, q4[v].x, acc[4 * v]);
            acc[4 * v + 1] = fmaf(w, q4[v].y, acc[4 * v + 1]);
            acc[4 * v + 2] = fmaf(w, q4[v].z, acc[4 * v + 2]);
            acc[4 * v + 3] = fmaf(w, q4[v].w, acc[4 * v + 3]);
          }
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          o0[e] = __float_as_uint(acc[e]);
          o1[e] = __float_as_uint(acc[32 + e]);
        }
      });
      if (row_ok && p.lse) p.lse[lse_index()] = lse_v;
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

template <int D, bool BF16>
cudaError_t launch_sk(const PrefillParams& p, int grid, cudaStream_t stream) {
  using L = SkLayout<D>;
  static std::atomic<uint64_t> smem_set{0};
  const cudaError_t e = ensure_dynamic_smem(prefill_sk_kernel<D, BF16>, L::kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  prefill_sk_kernel<D, BF16><<<grid, kThreads, L::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_streamk(const PrefillParams& p, int head_size, bool bf16, int grid,
                                   cudaStream_t stream) {
  if (head_size == 128) return bf16 ? launch_sk<128, true>(p, grid, stream) : launch_sk<128, false>(p, grid, stream);
  if (head_size == 64) return bf16 ? launch_sk<64, true>(p, grid, stream) : launch_sk<64, false>(p, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn

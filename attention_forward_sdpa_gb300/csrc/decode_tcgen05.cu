// decode_tcgen05.cu -- split-KV decode ("gfx942 unified attention, from the
// math up", sec. 8) for head sizes 64, 128 and 256 as a persistent, TMA-fed,
// tcgen05 kernel (the layout notes below are written for 128; 64 uses one
// channel half, 256 four halves and two O^T accumulators).  Decode is bound
// by HBM bandwidth (each K/V byte is read once and used for 2 * G flops), so
// the design goal is a continuous stream of page loads with as few
// instructions per byte as possible:
//
//   * A work item is (sequence, F consecutive KV heads, split) -- F KV heads
//     and all their query heads (F * G <= 16) at once, so that one TMA box
//     brings the same 16 page rows of F heads: with the cache viewed as
//     (channel, slot, head, page) a box of 64 channels x 16 slots x F heads
//     lands in shared memory as 16F consecutive 128-byte rows, and a 5-D view
//     (channel, slot, channel half, head, page) fetches both channel halves
//     of V in one instruction.  A 128-row key tile costs 3 * 8 / F TMA
//     instructions (6 for F = 4) instead of 32 with one head per item.
//   * Persistent CTAs (one per SM) claim items from an atomic counter in
//     longest-sequence-first order (each CTA ranks the sequence lengths it
//     caches in shared memory), so items balance dynamically.
//   * Warp 0 streams Q rows and page boxes into a 192 KB ring of 128-row
//     tiles (K and V alternate; six tiles of 32 KB at head size 128, twelve
//     of 16 KB at 64, three of 64 KB at 256); its lanes hold the page ids of
//     64 boxes at a time and issue the boxes in parallel.
//   * Warp 1 issues S^T = K Q^T (M = 128 tile rows, N = 16 query heads, fp32
//     in TMEM) and O^T += V^T P^T (M = 128 channels, N = 16).  P^T is block
//     diagonal (a row of KV head h only feeds the columns of h's query
//     heads); the off-diagonal zeros are written once.
//   * Warps 2-5 (one thread per tile row -- (box, KV head, key) -- then per
//     channel) take each tile's scores from TMEM, form the per-column running
//     max across the CTA (lazy: raised only when the tile's max exceeds it by
//     more than 8 in log2 units, which is exact and makes O rescales rare),
//     exp2, the running denominators, write P^T, rescale O^T when needed, and
//     at the end of an item write the partial state (un-normalised o, max in
//     log2 units, denominator) -- or, with one split, the rounded output.
//   * fp8 caches (E4M3 codes): TMA lands 128-byte rows of codes in staging
//     tiles, warps 6-9 widen each row exactly into the 16-bit ring tile the
//     MMAs read (one E4M3 byte per element is read from HBM instead of two);
//     the K factor is folded into tau, the V factor into the output.
// Every wait is bounded (see sm103_ptx.cuh); the CTA-wide exchange of the
// softmax warps also goes through an mbarrier so that it is bounded.

#include "attn_internal.h"
#include "e4m3.cuh"
#include "round16.cuh"
#include "score_features.cuh"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kRows = 128;              // tile rows: 16-key boxes x F heads x 16 keys
constexpr int kItemRing = 4;
constexpr int kHalfBytes = kRows * 128;         // K: 128 rows x 64 channels (one channel half)
constexpr int kPBytes = 2 * 16 * 128;           // two row halves of [16 heads][64 rows]
constexpr int kSortMax = 128;                   // longest-first order up to this many sequences
constexpr float kLn2 = 0.693147180559945309f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleSlack = 8.f;            // log2 units

struct ItemEntry {
  int b;       // sequence, or -1 at the end of the work
  int kvh0;    // first KV head of the item
  int q0;      // first query head of the item (column 0)
  int split;
  int k0, k1;  // key range
  int lo;      // first visible key (a sliding window masks the keys below)
  int sk;      // the sequence's KV length (its decode row is aligned with key sk - 1)
};

constexpr int kStage8Bytes = kRows * 128;      // an fp8 tile: 128 rows x 128 codes (16 KB)

// Shared-memory layout.  With 16-bit caches the ring holds 192 KB of tiles.  With
// fp8 caches (KV8) TMA lands the codes in four 16 KB staging tiles, four
// converter warps widen them into a ring of four 16-bit tiles (the layout
// the MMAs read), and the CTA has 320 threads instead of 192.
template <int D, bool KV8>
struct Lay {
  static_assert((D == 128 || D == 64 || D == 256) && (!KV8 || D == 128),
                "head size 128, or 64 / 256 with 16-bit caches");
  static constexpr int kD = D;
  static constexpr int kOBlocks = D == 256 ? 2 : 1;      // 128-channel blocks of O^T (TMEM)
  static constexpr int kSeqCache = D == 256 ? 1024 : 2048;   // cached sequence lengths
  static constexpr int kHalves = D / 64;                 // 64-channel halves of a row
  static constexpr int kTileBytes = kRows * D * 2;       // 16 / 32 / 64 KB at d = 64 / 128 / 256
  static constexpr int kQBytes = kHalves * 16 * 128;     // channel halves of [16 heads][64]
  static constexpr int kVGroup = kHalves * 2048;         // V: one 16-row group, all halves
  static constexpr int kThreads = KV8 ? 320 : 192;
  // 16-bit K/V ring slots of one tile each (about the same bytes in flight
  // at every head size: 12 x 16 KB, 6 x 32 KB, 3 x 64 KB)
  static constexpr int kSlots = KV8 ? 4 : (D == 64 ? 12 : (D == 256 ? 3 : 6));
  static constexpr int kStages = KV8 ? 4 : 0;    // fp8 staging slots
  static constexpr int kRingOff = 0;
  static constexpr int kStageOff = kRingOff + kSlots * kTileBytes;
  static constexpr int kQOff = kStageOff + kStages * kStage8Bytes;
  static constexpr int kPOff = kQOff + 2 * kQBytes;
  static constexpr int kRedOff = kPOff + 2 * kPBytes;          // float [2][8 groups][16]
  static constexpr int kLRedOff = kRedOff + 2 * 8 * 16 * 4;    // float [2][8 groups][16]
  static constexpr int kItemOff = kLRedOff + 2 * 8 * 16 * 4;   // ItemEntry [kItemRing]
  static constexpr int kSeqOff = kItemOff + kItemRing * (int)sizeof(ItemEntry);
  static constexpr int kOrderOff = kSeqOff + kSeqCache * 4;
  static constexpr int kFlagOff = kOrderOff + kSortMax * 4;    // int [3]
  static constexpr int kBarOff = kFlagOff + 16;
  // barriers: kv_full[kSlots] kv_empty[kSlots] q_full[2] q_empty[2] s_full[2]
  //           p_full[2] pv_done item_full[R] item_empty[R] mma_done red
  //           stage_full[kStages] stage_empty[kStages]
  static constexpr int kNumBars = 2 * kSlots + 2 + 2 + 2 + 2 + 1 + 2 * kItemRing + 1 + 1 +
                                  2 * kStages;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
};
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

// Byte offset of the 16-bit P^T element (column q, tile row r) in the
// K-major, 128-byte-swizzled B operand: two row halves of [16 columns][64].
__device__ __forceinline__ uint32_t p_offset(int q, int r) {
  const int half = r >> 6, c = r & 63;
  const int chunk = (c >> 3) ^ (q & 7);
  return (uint32_t)(half * 2048 + q * 128 + chunk * 16 + (c & 7) * 2);
}

template <bool BF16, int GH, bool KV8, int D>
__global__ void __launch_bounds__(Lay<D, KV8>::kThreads, 1) decode_tc_kernel(const __grid_constant__ DecodeParams p) {
  using L = Lay<D, KV8>;
  constexpr int kD = L::kD, kHalves = L::kHalves, kTileBytes = L::kTileBytes;
  constexpr int kQBytes = L::kQBytes, kVGroup = L::kVGroup, kOBlocks = L::kOBlocks;
  constexpr int kSeqCache = L::kSeqCache;
  constexpr int kThreads = L::kThreads, kSlots = L::kSlots, kStages = L::kStages;
  constexpr int kRingOff = L::kRingOff, kStageOff = L::kStageOff, kQOff = L::kQOff;
  constexpr int kPOff = L::kPOff, kRedOff = L::kRedOff, kLRedOff = L::kLRedOff;
  constexpr int kItemOff = L::kItemOff, kSeqOff = L::kSeqOff, kOrderOff = L::kOrderOff;
  constexpr int kFlagOff = L::kFlagOff, kBarOff = L::kBarOff, kMiscOff = L::kMiscOff;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sRing = base + kRingOff;
  const uint32_t sStage = base + kStageOff;
  const uint32_t sQ = base + kQOff;
  const uint32_t sP = base + kPOff;
  float* red = reinterpret_cast<float*>(smem + kRedOff);
  float* lred = reinterpret_cast<float*>(smem + kLRedOff);
  ItemEntry* items = reinterpret_cast<ItemEntry*>(smem + kItemOff);
  int* seq_cache = reinterpret_cast<int*>(smem + kSeqOff);
  int* order = reinterpret_cast<int*>(smem + kOrderOff);
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
  const uint32_t bar_st_full = bar_red + 8u;                 // fp8: staging tile landed
  const uint32_t bar_st_empty = bar_st_full + 8u * kStages;  // fp8: staging tile widened
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int F = p.kv_per_item;              // KV heads per item (GH * F <= 16)
  const int KT = kRows / F;                 // keys per tile
  // ALiBi raises the scores of the keys nearest the decode row, so walked in
  // key order the running maxima climb on every tile of a steep head (an O
  // rescale and a second CTA exchange each time).  With slopes each item
  // walks its tiles from the last to the first: the first tile then sets the
  // maxima, and the recurrence, exact in any order, rarely moves them.
  const bool rev = p.alibi != nullptr;
  const int BPT = KT / 16;                  // 16-key boxes per tile
  const int G = p.num_q_heads / p.num_kv_heads;
  const int subs = G / GH;                  // query-head groups per KV head (1 unless G > 16)
  const int groups = (p.num_kv_heads / F) * subs;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      // fp8: a ring tile is complete when the 128 converter threads arrive
      mbar_init(bar_kv_full + 8u * s, KV8 ? 128 : 1);
      mbar_init(bar_kv_empty + 8u * s, 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_st_full + 8u * s, 1);
      mbar_init(bar_st_empty + 8u * s, 128);
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
      mbar_init(bar_item_empty + 8u * i, 1 + 4 + (KV8 ? 4 : 0));
    }
    mbar_init(bar_mma_done, 1);
    mbar_init(bar_red, 128);
    for (int i = 0; i < 3; ++i) reinterpret_cast<volatile int*>(smem + kFlagOff)[i] = 0;
    *abort_flag = 0;
    fence_mbar_init();
  }
  // P^T is block diagonal: zero both buffers once; each softmax thread later
  // writes only its own (row, column) entries
  for (int i = threadIdx.x; i < 2 * kPBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + kPOff)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
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
    const bool cached = p.num_seqs <= kSeqCache;
    if (cached)
      for (int i = lane; i < p.num_seqs; i += 32) seq_cache[i] = p.seq_lens[i];
    __syncwarp();
    // longest sequences first (ties by index), so that the dynamic queue
    // ends with short items
    const bool sorted = cached && p.num_seqs <= kSortMax;
    if (sorted) {
      for (int b = lane; b < p.num_seqs; b += 32) {
        const int lb = seq_cache[b];
        int rank = 0;
        for (int c = 0; c < p.num_seqs; ++c) {
          const int lc = seq_cache[c];
          rank += (lc > lb || (lc == lb && c < b)) ? 1 : 0;
        }
        order[rank] = b;
      }
    }
    __syncwarp();
    // page ids of 64 boxes (1024 keys) at a time, two per lane: box q is held
    // by lane q % 32 in register q / 32, and that lane issues the box
    auto load_ids = [&](const int32_t* bt, int k0, int n_boxes, int cb, int (&pg)[2], int (&rw)[2]) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        pg[h] = 0;
        rw[h] = 0;
        const int q = cb + 32 * h + lane;
        if (q < n_boxes) {
          const int key = k0 + 16 * q;
          pg[h] = bt[key / bs];
          rw[h] = key % bs;
          if (pg[h] < 0 || pg[h] >= p.num_blocks) report_status(p.status, kStatusBadBlockTable);
        }
      }
    };
    for (;;) {
      int item = 0;
      if (lane == 0) item = atomicAdd(p.counter, 1);
      item = __shfl_sync(0xFFFFFFFFu, item, 0);
      const bool end = item >= p.n_items;
      int b = -1, kvh0 = 0, q0 = 0, split = 0, k0 = 0, k1 = 0, lo = 0, sk = 0;
      if (!end) {
        split = item % p.num_splits;
        const int rest = item / p.num_splits;
        const int grp = rest % groups;
        const int rank = rest / groups;
        b = sorted ? order[rank] : rank;
        kvh0 = (grp / subs) * F;
        q0 = kvh0 * G + (grp % subs) * GH;
        int Sk = cached ? seq_cache[b] : p.seq_lens[b];
        if (Sk < 0 || Sk > p.max_seqlen_k) {
          if (lane == 0) report_status(p.status, kStatusBadArg);
          Sk = 0;
        }
        // a sliding window keeps keys >= lo: the splits cut [lo rounded
        // down to 16, Sk), so boxes stay page-aligned, and the softmax masks
        // the keys below lo
        if (p.win_left >= 0) lo = max(0, Sk - 1 - p.win_left);
        sk = Sk;
        const int lo16 = lo & ~15;
        split_keys(Sk - lo16, p.num_splits, split, k0, k1);
        k0 += lo16;
        k1 += lo16;
      }
      const uint32_t rs = seen % kItemRing;
      if (seen >= kItemRing &&
          !mbar_wait(bar_item_empty + 8u * rs, ((seen / kItemRing) - 1) & 1, abort_flag))
        break;
      if (lane == 0) {
        ItemEntry e;
        e.b = b; e.kvh0 = kvh0; e.q0 = q0; e.split = split; e.k0 = k0; e.k1 = k1;
        e.lo = lo; e.sk = sk;
        items[rs] = e;
        mbar_arrive(bar_item_full + 8u * rs);
      }
      __syncwarp();
      ++seen;
      if (end) break;
      const int n_tiles = (k1 - k0 + KT - 1) / KT;
      if (n_tiles == 0) continue;
      // Q rows of the item's query heads
      const uint32_t qs = q_loads & 1u;
      if (q_loads >= 2 && !mbar_wait(bar_q_empty + 8u * qs, ((q_loads >> 1) - 1) & 1, abort_flag))
        break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_q_full + 8u * qs, (uint32_t)(kHalves * p.q_box_rows * 128));
        for (int h = 0; h < kHalves; ++h)
          tma_load_3d(sQ + qs * kQBytes + h * 2048, &p.tm_q, bar_q_full + 8u * qs, h * 64, q0, b);
      }
      ++q_loads;
      const int32_t* bt = p.block_table + (int64_t)b * p.bt_stride;
      const int n_boxes = (k1 - k0 + 15) / 16;
      bool ok = true;
      // the K and V boxes of one tile: nbox boxes from box rb of the 64-box
      // chunk whose page ids are in pg / rw (false when a wait ran out)
      auto issue_tile = [&](int rb, int nbox, const int (&pg)[2], const int (&rw)[2]) -> bool {
        const int set = rb >> 5;            // register holding this tile's ids
        const int j = lane - (rb & 31);     // this lane's box within the tile
        const bool mine = j >= 0 && j < nbox;
        const int page = set ? pg[1] : pg[0];
        const int row = set ? rw[1] : rw[0];
        for (int kind = 0; kind < 2; ++kind) {
          if constexpr (KV8) {
            // fp8: one box of 128 codes x 16 slots x F heads per 16 keys
            // lands as 16F rows of 128 bytes in a staging tile
            const uint32_t s8 = fills % kStages;
            if (fills >= kStages &&
                !mbar_wait(bar_st_empty + 8u * s8, ((fills / kStages) - 1) & 1, abort_flag))
              return false;
            const uint32_t bar = bar_st_full + 8u * s8;
            if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(nbox * F * 2048));
            __syncwarp();
            if (mine)
              tma_load_4d(sStage + s8 * kStage8Bytes + j * F * 2048, kind == 0 ? &p.tm_k : &p.tm_v,
                          bar, 0, row, kvh0, page);
            last_fill[s8] = fills + 1;
            ++fills;
            continue;
          }
          const uint32_t s = fills % kSlots;
          if (fills >= kSlots &&
              !mbar_wait(bar_kv_empty + 8u * s, ((fills / kSlots) - 1) & 1, abort_flag))
            return false;
          const uint32_t bar = bar_kv_full + 8u * s;
          if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(nbox * F * kVGroup));
          __syncwarp();
          if (mine) {
            const uint32_t slot = sRing + s * kTileBytes;
            if (kind == 0) {
              // K: [channel half][tile row], box j -> rows [16 F j, 16 F (j + 1))
              const uint32_t dst = slot + j * F * 16 * 128;
#pragma unroll
              for (int h = 0; h < kHalves; ++h)
                tma_load_4d(dst + h * kHalfBytes, &p.tm_k, bar, 64 * h, row, kvh0, page);
            } else {
              // V: [16-row group][channel half][16 rows], both halves at once
              tma_load_5d(slot + j * F * kVGroup, &p.tm_v, bar, 0, row, 0, kvh0, page);
            }
          }
          last_fill[s] = fills + 1;
          ++fills;
        }
        return true;
      };
      if (!rev) {
        // key order: chunk by chunk of 64 boxes, tile by tile
        for (int cb = 0; cb < n_boxes && ok; cb += 64) {
          int pg[2], rw[2];
          load_ids(bt, k0, n_boxes, cb, pg, rw);
          const int chunk_boxes = min(64, n_boxes - cb);
          for (int rb = 0; rb < chunk_boxes && ok; rb += BPT)
            ok = issue_tile(rb, min(BPT, chunk_boxes - rb), pg, rw);
        }
      } else {
        // ALiBi: the last tile first (a tile's BPT boxes never straddle a
        // 64-box chunk of page ids; a chunk is loaded when a tile enters it)
        int loaded_cb = -1;
        int pg[2] = {0, 0}, rw[2] = {0, 0};
        for (int w = 0; w < n_tiles && ok; ++w) {
          const int box0 = (n_tiles - 1 - w) * BPT;   // the tile's first box
          const int cb = box0 & ~63;
          if (cb != loaded_cb) {
            load_ids(bt, k0, n_boxes, cb, pg, rw);
            loaded_cb = cb;
          }
          ok = issue_tile(box0 - cb, min(BPT, n_boxes - box0), pg, rw);
        }
      }
      if (!ok) break;
    }
    // no copy may still be in flight into this CTA's shared memory
    if (lane == 0) {
      // (fp8: the copies go to the staging tiles)
      constexpr int kN = KV8 ? kStages : kSlots;
      const uint32_t full = KV8 ? bar_st_full : bar_kv_full;
      for (int s = 0; s < kN; ++s)
        if (last_fill[s] > 0) drain_wait(full + 8u * s, (last_fill[s] - 1) / kN & 1);
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
        for (int ob = 0; ob < kOBlocks; ++ob)
#pragma unroll
          for (int kk = 0; kk < kRows / 16; ++kk) {
            // A = V^T (MN-major): 16 rows per step, channel halves 2048 B
            // apart; O^T block ob (channels 128 ob .. 128 ob + 127, TMEM
            // columns kOCol + 16 ob) starts at channel half 2 ob.  At d = 64
            // the product still has M = 128: its rows 64-127 read the next
            // 16-row group (finite or not), land in O^T rows that are never
            // stored, and never touch rows 0-63.
            umma_ss(tmem + kOCol + 16u * ob,
                    make_sdesc_sw128(a0 + kk * kVGroup + ob * 4096, 2048, 1024),
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
      const int n_tiles = (e.k1 - e.k0 + KT - 1) / KT;
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
  } else if (!KV8 || warp < 6) {
    // ---------------------------------------------------------- softmax + epilogue
    const int quarter = warp & 3;            // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;       // tile row (S^T) / channel (O^T)
    const int grp16 = r >> 4;                // (box, head) group of the row: box * F + head
    const int hrow = grp16 % F;              // KV head of the row within the item
    const int krow = (grp16 / F) * 16 + (r & 15);   // key of the row within the tile
    const int c0 = hrow * GH;                // first column of the row's query heads
    const int NC = F * GH;                   // columns in use
    const int NG = kRows / 16;               // (box, head) groups per tile
    constexpr int SW = GH == 16 ? 16 : 2 * GH;   // score columns loaded per warp
    const int cwin = F >= 2 ? ((2 * quarter) % F) * GH : 0;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    const float inv_cap = p.softcap > 0.f ? 1.f / p.softcap : 0.f;
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
      const int n_tiles = (e.k1 - e.k0 + KT - 1) / KT;
      // query head of the row's column j is qbase + j
      const int qbase = (e.kvh0 + hrow) * G + (e.q0 - e.kvh0 * G);
      float slope[GH];
#pragma unroll
      for (int j = 0; j < GH; ++j) slope[j] = p.alibi ? p.alibi[qbase + j] : 0.f;
      float mcol[16];   // running max of every column (kept identically by all threads)
#pragma unroll
      for (int c = 0; c < 16; ++c) mcol[c] = -INFINITY;
      // running max of the row's own columns (identical in every thread of
      // the same KV head), partial denominators of this thread's keys
      float m[GH], lp[GH];
#pragma unroll
      for (int j = 0; j < GH; ++j) {
        m[j] = -INFINITY;
        lp[j] = 0.f;
      }
      for (int t = 0; t < n_tiles && ok; ++t) {
        if (!mbar_wait(bar_s_full + 8u * (g & 1u), (g >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        // the warp's rows belong to one KV head (F = 1) or two adjacent ones:
        // load their 2 * GH columns and keep this lane's half
        uint32_t sv[SW];
        tmem_ld_n<SW>(tmem + lane_off + s_col(g) + cwin, sv);
        tmem_ld_wait_n<SW>(sv);
        const int key = e.k0 + (rev ? n_tiles - 1 - t : t) * KT + krow;
        const bool valid = key >= e.lo && key < e.k1;
        const bool upper = SW > GH && F >= 2 && lane >= 16;
        float x[GH];
        bool raise = false;
#pragma unroll
        for (int j = 0; j < GH; ++j) {
          const float v = __uint_as_float(upper ? sv[(GH + j) % SW] : sv[j]);
          if (p.score_xform) {
            // softcap, then ALiBi on the scaled score; distance to the
            // decode row's aligned key
            const float xs = rewrite_score(v * p.scale, p.softcap, inv_cap, slope[j],
                                           (float)(e.sk - 1 - key));
            x[j] = valid ? xs * kLog2e : -INFINITY;
          } else {
            x[j] = valid ? v * sl2 : -INFINITY;
          }
          raise |= x[j] > m[j] + kRescaleSlack;
        }
        // Announce before the exchange whether any score of this tile exceeds
        // its column's running max by more than the slack: only then does the
        // max move (and O^T need a rescale).  Flags rotate over three words;
        // the word for tile t + 1 is cleared here, before anyone can pass
        // this tile's exchange and write it.
        volatile int* flags = reinterpret_cast<volatile int*>(smem + kFlagOff);
        const uint32_t fi = red_uses % 3u;
        if (r == 0) flags[(fi + 1u) % 3u] = 0;
        if (t == 0 || raise) flags[fi] = 1;
        if (!cta_sync()) { ok = false; break; }
        const bool heavy = flags[fi] != 0;
        float alpha_own[GH];
#pragma unroll
        for (int j = 0; j < GH; ++j) alpha_own[j] = 1.f;
        bool rescale = false;
        float alpha_all[16];
        if (heavy) {
          // the tile max of every column: 16-key maxima of each (box, head)
          // group, then across boxes
          float* rb = red + (red_uses & 1u) * 128;
#pragma unroll
          for (int j = 0; j < GH; ++j) {
            float v = x[j];
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
            if ((lane & 15) == 0) rb[grp16 * 16 + j] = v;
          }
          if (!cta_sync()) { ok = false; break; }
#pragma unroll
          for (int c = 0; c < 16; ++c) alpha_all[c] = 1.f;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            if (c >= NC) break;
            const int hh = c / GH, jj = c % GH;
            float tm = -INFINITY;
            for (int gg = hh; gg < NG; gg += F) tm = fmaxf(tm, rb[gg * 16 + jj]);
            const float mo = mcol[c];
            const float mn = (tm > mo + kRescaleSlack || mo == -INFINITY) ? fmaxf(tm, mo) : mo;
            const float a = mo == -INFINITY ? 0.f : fast_exp2(mo - mn);
            if (c / GH == hrow) {
#pragma unroll
              for (int j = 0; j < GH; ++j)
                if (j == jj) {
                  alpha_own[j] = a;
                  m[j] = mn;
                }
            }
#pragma unroll
            for (int cc = 0; cc < 16; ++cc)
              if (cc == c) alpha_all[cc] = a;
            rescale |= a != 1.f;
            mcol[c] = mn;
          }
        }
        float pr[GH];
#pragma unroll
        for (int j = 0; j < GH; ++j) {
          const float mu = m[j] == -INFINITY ? 0.f : m[j];
          pr[j] = fast_exp2(x[j] - mu);
          lp[j] = fmaf(lp[j], alpha_own[j], pr[j]);
        }
        // PV of the previous tile must be complete before O^T and the P^T
        // buffer of two tiles ago are touched
        if (g >= 1) {
          if (!mbar_wait(bar_pv_done, (g - 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
        }
        if (t > 0 && heavy && rescale) {
#pragma unroll
          for (int ob = 0; ob < kOBlocks; ++ob) {
            uint32_t ov[16];
            tmem_ld16(tmem + lane_off + kOCol + 16u * ob, ov);
            tmem_ld_wait_n<16>(ov);
#pragma unroll
            for (int c = 0; c < 16; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha_all[c]);
            tmem_st16(tmem + lane_off + kOCol + 16u * ob, ov);
          }
          tmem_st_wait();
        }
        if (!valid) {
          // this row's V may hold another split's key, a stale tile or poison:
          // P is 0 there, but 0 * NaN is not, so zero the row
          const uint32_t fill_v = 2u * g + 1u;
          const uint32_t sv_slot = fill_v % kSlots;
          if (!mbar_wait(bar_kv_full + 8u * sv_slot, (fill_v / kSlots) & 1, abort_flag)) { ok = false; break; }
          uint8_t* vrow = smem + (sRing - base) + sv_slot * kTileBytes + grp16 * kVGroup + (r & 15) * 128;
#pragma unroll
          for (int h = 0; h < kHalves; ++h)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(vrow + h * 2048 + c * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        uint8_t* pb = smem + (sP - base) + (g & 1u) * kPBytes;
#pragma unroll
        for (int j = 0; j < GH; ++j) {
          const uint16_t v = BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(pr[j]))
                                  : __half_as_ushort(__float2half_rn(pr[j]));
          *reinterpret_cast<uint16_t*>(pb + p_offset(c0 + j, r)) = v;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar_p_full + 8u * (g & 1u));
        ++g;
      }
      if (!ok) break;
      // ---- item epilogue: denominators, then partial or final output
      float o[kOBlocks][16];   // O^T rows r and (d = 256) r + 128
      if (n_tiles > 0) {
        if (!mbar_wait(bar_pv_done, (g - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int ob = 0; ob < kOBlocks; ++ob) {
          uint32_t ov[16];
          tmem_ld16(tmem + lane_off + kOCol + 16u * ob, ov);
          tmem_ld_wait_n<16>(ov);
#pragma unroll
          for (int c = 0; c < 16; ++c) o[ob][c] = __uint_as_float(ov[c]);
        }
      } else {
#pragma unroll
        for (int ob = 0; ob < kOBlocks; ++ob)
#pragma unroll
          for (int c = 0; c < 16; ++c) o[ob][c] = 0.f;
      }
      float* lb = lred + (red_uses & 1u) * 128;
#pragma unroll
      for (int j = 0; j < GH; ++j) {
        float v = lp[j];
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        if ((lane & 15) == 0) lb[grp16 * 16 + j] = v;
      }
      if (!cta_sync()) { ok = false; break; }
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        if (c >= NC) break;
        const int hh = c / GH, jj = c % GH;
        float L = 0.f;
        for (int gg = hh; gg < NG; gg += F) L += lb[gg * 16 + jj];
        const int qh = (e.kvh0 + hh) * G + (e.q0 - e.kvh0 * G) + jj;
        const int64_t row = (int64_t)e.b * Hq + qh;
        if (p.num_splits > 1) {
#pragma unroll
          for (int ob = 0; ob < kOBlocks; ++ob)
            if (r + 128 * ob < kD) p.part_o[(row * p.num_splits + e.split) * kD + r + 128 * ob] = o[ob][c];
          if (r == 0) {
            p.part_ml[(row * p.num_splits + e.split) * 2 + 0] = mcol[c];
            p.part_ml[(row * p.num_splits + e.split) * 2 + 1] = L;
          }
        } else {
          // one split: normalise here, with the sink logit in the
          // denominator when the call has one
          float inv_l, lse_v;
          finish_row(mcol[c], L, p.sinks ? p.sinks[qh] : -INFINITY, inv_l, lse_v);
#pragma unroll
          for (int ob = 0; ob < kOBlocks; ++ob) {
            const int ch = r + 128 * ob;
            const float v = o[ob][c] * (inv_l * p.out_scale);   // fp8 V factor (1 otherwise)
            if (ch < kD) {   // O^T rows past the head size are not part of the result
              if (p.rounding == 3) static_cast<float*>(p.out)[row * kD + ch] = v;
              else static_cast<uint16_t*>(p.out)[row * kD + ch] = round_out<BF16>(v, p.rounding);
            }
          }
          if (r == 0 && p.lse) p.lse[row] = lse_v;
        }
      }
    }
    tc_fence_before();
  } else {
    // ---------------------------------------------------------- fp8 converters
    // Warps 6-9 (fp8 caches only): thread t widens row t of each staging
    // tile (128 E4M3 codes, exact in bf16 / fp16) into ring tile `fills %
    // kSlots` in the MMA's 128-byte-swizzled layout: K as [channel half][row],
    // V as [16-row group][channel half][row % 16].  Fills alternate K, V.
    if constexpr (KV8) {
      const int t = threadIdx.x - 6 * 32;
      const uint32_t sw = (uint32_t)(t & 7);   // swizzle phase of the row (same on both sides)
      uint32_t seen = 0, fills = 0;
      bool ok = true;
      for (;;) {
        const uint32_t rs = seen % kItemRing;
        if (!mbar_wait(bar_item_full + 8u * rs, (seen / kItemRing) & 1, abort_flag)) break;
        const ItemEntry e = items[rs];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_item_empty + 8u * rs);
        ++seen;
        if (e.b < 0) break;
        const int n_fills = 2 * ((e.k1 - e.k0 + KT - 1) / KT);
        for (int f = 0; f < n_fills; ++f, ++fills) {
          const uint32_t s8 = fills % kStages, sr = fills % kSlots;
          if (!mbar_wait(bar_st_full + 8u * s8, (fills / kStages) & 1, abort_flag)) { ok = false; break; }
          if (fills >= kSlots &&
              !mbar_wait(bar_kv_empty + 8u * sr, ((fills / kSlots) - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const uint8_t* src = smem + kStageOff + s8 * kStage8Bytes + t * 128;
          uint8_t* dst = smem + kRingOff + sr * kTileBytes;
          const bool is_v = (fills & 1u) != 0;
          uint8_t* row0 = is_v ? dst + (t >> 4) * 4096 + (t & 15) * 128 : dst + t * 128;
          const int half_stride = is_v ? 2048 : kHalfBytes;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 w = *reinterpret_cast<const uint4*>(src + ((c ^ sw) << 4));
            uint4 lo, hi;
            e4m3x16_widen<BF16>(w, lo, hi);
            uint8_t* hrow = row0 + (c >> 2) * half_stride;
            const uint32_t c0 = 2u * (c & 3);
            *reinterpret_cast<uint4*>(hrow + ((c0 ^ sw) << 4)) = lo;
            *reinterpret_cast<uint4*>(hrow + (((c0 + 1u) ^ sw) << 4)) = hi;
          }
          // every thread publishes its own row to the tensor core's proxy
          fence_proxy_async_smem();
          mbar_arrive(bar_st_empty + 8u * s8);
          mbar_arrive(bar_kv_full + 8u * sr);
        }
        if (!ok) break;
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) report_status(p.status, kStatusTimeout);
}

template <bool BF16, int GH, bool KV8, int D>
cudaError_t launch_k(const DecodeParams& p, int grid, cudaStream_t stream) {
  using L = Lay<D, KV8>;
  static std::atomic<uint64_t> smem_set{0};
  const cudaError_t e = ensure_dynamic_smem(decode_tc_kernel<BF16, GH, KV8, D>, L::kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  decode_tc_kernel<BF16, GH, KV8, D><<<grid, L::kThreads, L::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

template <bool BF16, int GH>
cudaError_t launch_t(const DecodeParams& p, int head_size, int grid, cudaStream_t stream) {
  if (head_size == 64 || head_size == 256) {
    if (p.kv_fp8) return cudaErrorInvalidValue;   // fp8 at d = 64 / 256 takes the SIMT kernel
    return head_size == 64 ? launch_k<BF16, GH, false, 64>(p, grid, stream)
                           : launch_k<BF16, GH, false, 256>(p, grid, stream);
  }
  return p.kv_fp8 ? launch_k<BF16, GH, true, 128>(p, grid, stream)
                  : launch_k<BF16, GH, false, 128>(p, grid, stream);
}

template <bool BF16>
cudaError_t launch_b(const DecodeParams& p, int head_size, int grid, cudaStream_t stream) {
  switch (p.heads_per_item) {
    case 1: return launch_t<BF16, 1>(p, head_size, grid, stream);
    case 2: return launch_t<BF16, 2>(p, head_size, grid, stream);
    case 4: return launch_t<BF16, 4>(p, head_size, grid, stream);
    case 8: return launch_t<BF16, 8>(p, head_size, grid, stream);
    case 16: return launch_t<BF16, 16>(p, head_size, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// Splits of one decode step on the tcgen05 path (head size 128).  The caller
// has chosen heads_per_item (query heads per KV head in an item: G, or 16
// when G is a multiple of 16 above it; a power of two) and kv_per_item (F,
// with F * heads_per_item <= 16 and F dividing num_kv_heads), encoded the
// tensor maps and zeroed p.counter on `stream`.
cudaError_t launch_decode_tc(const DecodeParams& p, int head_size, bool bf16, int grid,
                             cudaStream_t stream) {
  return bf16 ? launch_b<true>(p, head_size, grid, stream) : launch_b<false>(p, head_size, grid, stream);
}

}  // namespace attn

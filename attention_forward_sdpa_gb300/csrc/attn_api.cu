// attn_api.cu -- the extern "C" boundary declared in include/attn_fwd.h:
// argument validation (all on the host, before any launch), device check,
// TMA descriptor encoding (through a cache of descriptors) and grid sizing for
// attn_fwd_prefill, attn_fwd_dense, attn_fwd_decode, their feature-flagged
// (_ex) forms and the timeout test hook.  Every compute step runs in the
// kernels of prefill_tcgen05.cu, prefill_d256_tcgen05.cu, decode_tcgen05.cu,
// decode_splitkv.cu and kv_widen.cu.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <atomic>
#include <chrono>
#include <cstring>
#include <mutex>
#include <random>

#include "../../include/attn_fwd.h"
#include "attn_internal.h"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// The kernels are built for sm_103a only.
attn_status_t check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (major != 10 || minor != 3) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

constexpr uint64_t kDefaultWaitLimitNs = 4000000000ull;   // 4 s per pipeline wait

// Call numbers that tag the split prefill's merge tickets: a process-wide
// counter that starts at a random 48-bit value, so that tickets left in a
// workspace by earlier calls (or by nothing: fresh memory) do not match.
uint64_t next_call_epoch() {
  static std::atomic<uint64_t> counter{[] {
    std::random_device rd;
    const uint64_t t = (uint64_t)std::chrono::steady_clock::now().time_since_epoch().count();
    return ((uint64_t)rd() << 32 ^ (uint64_t)rd() ^ t * 0x9E3779B97F4A7C15ull) & 0xFFFFFFFFFFFFull;
  }()};
  return counter.fetch_add(1, std::memory_order_relaxed) + 1;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// int32 and fp32 arrays (NULL passes: optional arrays are checked for NULL
// where they are required)
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool valid_scale(float s) { return std::isfinite(s) && s > 0.f; }

constexpr float kLog2e = 1.4426950408889634f;

// The feature flags of attn_features_t, validated (NULL = none).
struct Features {
  int32_t win_left = -1, win_right = -1;
  float softcap = 0.f;
  const float* alibi = nullptr;
  const float* sinks = nullptr;
  bool kv_fp8 = false;
  float k_scale = 1.f, v_scale = 1.f;
  void* workspace = nullptr;
  size_t workspace_bytes = 0;
};

attn_status_t read_features(const attn_features_t* f, Features& out) {
  out = Features();
  if (!f) return ATTN_OK;
  if (f->window_left < -1 || f->window_right < -1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(f->softcap) || f->softcap < 0.f) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(f->alibi_slopes) & 3u) ||
      (reinterpret_cast<uintptr_t>(f->sinks) & 3u))
    return ATTN_ERR_INVALID_ARG;
  out.win_left = f->window_left;
  out.win_right = f->window_right;
  out.softcap = f->softcap;
  out.alibi = f->alibi_slopes;
  out.sinks = f->sinks;
  if (f->kv_fp8 != 0 && f->kv_fp8 != 1) return ATTN_ERR_INVALID_ARG;
  if (f->kv_fp8) {
    if (!valid_scale(f->k_scale) || !valid_scale(f->v_scale)) return ATTN_ERR_INVALID_ARG;
    out.kv_fp8 = true;
    out.k_scale = f->k_scale;
    out.v_scale = f->v_scale;
    out.workspace = f->workspace;
    out.workspace_bytes = f->workspace_bytes;
  }
  return ATTN_OK;
}

// Layout of the fp8 prefill workspace: widened K pages, widened V pages,
// block table, each at a 256-byte boundary.
struct Fp8Workspace {
  size_t k_off, v_off, table_off, total;
  int64_t pages_per_seq, n_pages, page_elems;
};

bool fp8_workspace_layout(int32_t num_seqs, int32_t max_seqlen_k, int32_t num_kv_heads,
                          int32_t head_size, int32_t block_size, Fp8Workspace& w) {
  if (num_seqs <= 0 || max_seqlen_k < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0)
    return false;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  w.pages_per_seq = ((int64_t)max_seqlen_k + block_size - 1) / block_size;
  if (w.pages_per_seq < 1) w.pages_per_seq = 1;
  w.n_pages = (int64_t)num_seqs * w.pages_per_seq;
  w.page_elems = (int64_t)block_size * num_kv_heads * head_size;
  const size_t cache_bytes = up((size_t)w.n_pages * (size_t)w.page_elems * 2);
  w.k_off = 0;
  w.v_off = cache_bytes;
  w.table_off = 2 * cache_bytes;
  w.total = w.table_off + up((size_t)w.n_pages * 4);
  return true;
}

void set_features(attn::PrefillParams& p, const Features& f, float scale) {
  p.win_left = f.win_left;
  p.win_right = f.win_right;
  p.softcap = f.softcap;
  p.alibi = f.alibi;
  p.sinks = f.sinks;
  p.scale = scale;
  p.score_xform = (f.softcap > 0.f || f.alibi) ? 1 : 0;
  p.out_scale = f.kv_fp8 ? f.v_scale : 1.f;
}

// Prefill grid (x: head units, z: row units; y is the sequence).  Head sizes
// 64 and 128 put two 128-row query tiles in a CTA: two heads of a GQA group
// when the group size is even, else two row blocks of one head.  Head size
// 256 has one query tile per CTA.
void prefill_grid(int head_size, bool pair_heads, int num_q_heads, int64_t row_blocks, int64_t& gx,
                  int64_t& gz) {
  if (head_size == 256) {
    gx = num_q_heads;
    gz = row_blocks;
  } else {
    gx = pair_heads ? num_q_heads / 2 : num_q_heads;
    gz = pair_heads ? row_blocks : (row_blocks + 1) / 2;
  }
}

}  // namespace

namespace attn {

namespace {

// Tensor-map cache.  A CUtensorMap is a pure function of the arguments of
// cuTensorMapEncodeTiled (base address, element type, sizes, strides, box,
// swizzle), so an entry keyed on all of them stays valid for as long as the
// process runs, whatever happened to the memory in between: a buffer freed and
// allocated again at the same address with the same shape encodes to the same
// map.  The cache saves the host-side encode of repeated calls (a serving
// loop calls with the same cache pool and, usually, the same activation
// buffers).  4-way set associative with LRU replacement (64 sets), so the
// four descriptors of one call never evict one another; one mutex.
struct MapKey {
  const void* base;
  uint32_t dtype, rank, swz, pad;
  cuuint64_t dims[5];
  cuuint64_t strides[4];
  cuuint32_t box[5];
  uint32_t pad2;
};

struct MapEntry {
  bool valid;
  uint64_t used;     // last use (a global tick), for LRU replacement
  MapKey key;
  CUtensorMap map;
};

constexpr int kMapSets = 64, kMapWays = 4;
std::mutex g_map_mutex;
MapEntry g_map_cache[kMapSets][kMapWays];
uint64_t g_map_tick = 0;
std::atomic<uint64_t> g_map_hits{0}, g_map_misses{0};

uint64_t key_hash(const MapKey& k) {
  // FNV-1a over the key's bytes
  const unsigned char* b = reinterpret_cast<const unsigned char*>(&k);
  uint64_t h = 1469598103934665603ull;
  for (size_t i = 0; i < sizeof(MapKey); ++i) h = (h ^ b[i]) * 1099511628211ull;
  return h;
}

bool encode_cached(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const cuuint64_t* dims,
                   const cuuint64_t* strides_bytes, const cuuint32_t* box, const void* base,
                   CUtensorMapSwizzle swz) {
  if (rank < 1 || rank > 5) return false;
  MapKey k;
  std::memset(&k, 0, sizeof(k));
  k.base = base;
  k.dtype = (uint32_t)dtype;
  k.rank = (uint32_t)rank;
  k.swz = (uint32_t)swz;
  for (int i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
    if (i + 1 < rank) k.strides[i] = strides_bytes[i];
  }
  MapEntry* set = g_map_cache[key_hash(k) % kMapSets];
  {
    std::lock_guard<std::mutex> lock(g_map_mutex);
    for (int w = 0; w < kMapWays; ++w) {
      MapEntry& e = set[w];
      if (e.valid && std::memcmp(&e.key, &k, sizeof(k)) == 0) {
        e.used = ++g_map_tick;
        *map = e.map;
        g_map_hits.fetch_add(1, std::memory_order_relaxed);
        return true;
      }
    }
  }
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  if (fn(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), dims, strides_bytes, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  g_map_misses.fetch_add(1, std::memory_order_relaxed);
  std::lock_guard<std::mutex> lock(g_map_mutex);
  int victim = 0;
  for (int w = 0; w < kMapWays; ++w) {
    if (!set[w].valid) { victim = w; break; }
    if (set[w].used < set[victim].used) victim = w;
  }
  MapEntry& e = set[victim];
  e.valid = true;
  e.used = ++g_map_tick;
  e.key = k;
  e.map = *map;
  return true;
}

}  // namespace

bool encode_tiled(CUtensorMap* map, bool bf16, int rank, const cuuint64_t* dims,
                  const cuuint64_t* strides_bytes, const cuuint32_t* box, const void* base,
                  CUtensorMapSwizzle swz) {
  return encode_cached(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                       rank, dims, strides_bytes, box, base, swz);
}

bool encode_tiled_u8(CUtensorMap* map, int rank, const cuuint64_t* dims,
                     const cuuint64_t* strides_bytes, const cuuint32_t* box, const void* base,
                     CUtensorMapSwizzle swz) {
  return encode_cached(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, dims, strides_bytes, box, base, swz);
}

int device_sm_count() {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Workspace: [partial o: rows * splits * d fp32][partial (m, l): rows * splits
// * 2 fp32][work counter, 256 bytes].
int decode_prepare_and_launch(DecodeParams& p, int head_size, bool bf16, void* workspace,
                              cudaStream_t stream) {
  const size_t rows = (size_t)p.num_seqs * (size_t)p.num_q_heads * (size_t)p.num_splits;
  float* ws = static_cast<float*>(workspace);
  const size_t counter_bytes = 256;
  if (p.num_splits > 1) {
    p.part_o = ws;
    p.part_ml = ws + rows * (size_t)head_size;
    p.counter = reinterpret_cast<int32_t*>(p.part_ml + rows * 2);
  } else {
    p.part_o = nullptr;
    p.part_ml = nullptr;
    p.counter = reinterpret_cast<int32_t*>(ws);
  }
  const int G = p.num_q_heads / p.num_kv_heads;
  const bool pow2 = (G & (G - 1)) == 0;
  // tcgen05 kernel: head size 128, or 64 / 256 with 16-bit caches
  const bool tc_path = (head_size == 128 || ((head_size == 64 || head_size == 256) && !p.kv_fp8)) &&
                       ((G <= 16 && pow2) || G % 16 == 0);
  if (!tc_path) {
    cudaError_t e = launch_decode(p, head_size, bf16, G, stream);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  p.heads_per_item = G <= 16 ? G : 16;
  // KV heads per item: as many as divide Hkv, fit 16 query-head columns, <= 4
  p.kv_per_item = 1;
  for (int f = 4; f > 1; f >>= 1)
    if (p.num_kv_heads % f == 0 && f * p.heads_per_item <= 16) {
      p.kv_per_item = f;
      break;
    }
  p.q_box_rows = p.num_q_heads < 16 ? p.num_q_heads : 16;
  const int64_t n_items = (int64_t)p.num_seqs * (p.num_kv_heads / p.kv_per_item) *
                          (G / p.heads_per_item) * (int64_t)p.num_splits;
  if (n_items > 2147483647) return ATTN_ERR_UNSUPPORTED;
  p.n_items = (int32_t)n_items;
  const cuuint64_t d = (cuuint64_t)head_size;
  const cuuint64_t slot_stride = d * 2 * (cuuint64_t)p.num_kv_heads;
  const cuuint64_t block_stride = slot_stride * (cuuint64_t)p.block_size;
  if (p.kv_fp8) {
    // fp8 codes as (channel, slot, head, page): a box of all 128 codes x 16
    // slots x F heads lands as 16F rows of 128 bytes (K and V alike)
    const cuuint64_t dims[4] = {d, (cuuint64_t)p.block_size, (cuuint64_t)p.num_kv_heads,
                                (cuuint64_t)p.num_blocks};
    const cuuint64_t strides[3] = {d * (cuuint64_t)p.num_kv_heads, d,
                                   d * (cuuint64_t)p.num_kv_heads * (cuuint64_t)p.block_size};
    const cuuint32_t box[4] = {128, 16, (cuuint32_t)p.kv_per_item, 1};
    if (!encode_tiled_u8(&p.tm_k, 4, dims, strides, box, p.k_cache, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled_u8(&p.tm_v, 4, dims, strides, box, p.v_cache, CU_TENSOR_MAP_SWIZZLE_128B))
      return ATTN_ERR_CUDA;
  }
  {
    const cuuint64_t dims[3] = {d, (cuuint64_t)p.num_q_heads, (cuuint64_t)p.num_seqs};
    const cuuint64_t strides[2] = {d * 2, d * 2 * (cuuint64_t)p.num_q_heads};
    const cuuint32_t box[3] = {64, (cuuint32_t)p.q_box_rows, 1};
    if (!encode_tiled(&p.tm_q, bf16, 3, dims, strides, box, p.q, CU_TENSOR_MAP_SWIZZLE_128B))
      return ATTN_ERR_CUDA;
  }
  if (!p.kv_fp8) {
    // K as (channel, slot, head, page): a box of 16 slots x F heads lands as
    // 16F consecutive rows of 64 channels
    const cuuint64_t dims[4] = {d, (cuuint64_t)p.block_size, (cuuint64_t)p.num_kv_heads,
                                (cuuint64_t)p.num_blocks};
    const cuuint64_t strides[3] = {slot_stride, d * 2, block_stride};
    const cuuint32_t box[4] = {64, 16, (cuuint32_t)p.kv_per_item, 1};
    if (!encode_tiled(&p.tm_k, bf16, 4, dims, strides, box, p.k_cache, CU_TENSOR_MAP_SWIZZLE_128B))
      return ATTN_ERR_CUDA;
  }
  if (!p.kv_fp8) {
    // V as (channel in half, slot, channel half, head, page): one box brings
    // both channel halves of 16 slots x F heads
    const cuuint64_t dims[5] = {64, (cuuint64_t)p.block_size, d / 64, (cuuint64_t)p.num_kv_heads,
                                (cuuint64_t)p.num_blocks};
    const cuuint64_t strides[4] = {slot_stride, 128, d * 2, block_stride};
    const cuuint32_t box[5] = {64, 16, (cuuint32_t)(d / 64), (cuuint32_t)p.kv_per_item, 1};
    if (!encode_tiled(&p.tm_v, bf16, 5, dims, strides, box, p.v_cache, CU_TENSOR_MAP_SWIZZLE_128B))
      return ATTN_ERR_CUDA;
  }
  const int sms = device_sm_count();
  if (sms <= 0) return ATTN_ERR_CUDA;
  const int grid = (int)(n_items < sms ? n_items : sms);
  if (cudaMemsetAsync(p.counter, 0, counter_bytes, stream) != cudaSuccess) return ATTN_ERR_CUDA;
  cudaError_t e = launch_decode_tc(p, head_size, bf16, grid, stream);
  if (e == cudaSuccess && p.num_splits > 1) e = launch_decode_combine(p, head_size, bf16, stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int check_decode_args(const void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_table, int32_t block_table_stride,
                      const int32_t* seq_lens, int32_t num_seqs, int32_t max_seqlen_k,
                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                      int32_t block_size, int32_t num_blocks, float scale, int32_t num_splits,
                      int dtype, int rounding, const float* lse_out, const int32_t* status_dev,
                      bool* empty) {
  *empty = false;
  if (num_seqs < 0 || max_seqlen_k < 0) return ATTN_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (rounding < ATTN_RTNE || rounding > ATTN_OUT_F32) return ATTN_ERR_INVALID_ARG;
  if (!valid_scale(scale)) return ATTN_ERR_INVALID_ARG;
  if (block_size <= 0 || num_blocks <= 0) return ATTN_ERR_INVALID_ARG;
  if (num_splits < 1 || num_splits > 64) return ATTN_ERR_INVALID_ARG;
  if (head_size != 64 && head_size != 128 && head_size != 256) return ATTN_ERR_UNSUPPORTED;
  if (block_size % 16 != 0) return ATTN_ERR_UNSUPPORTED;
  if (num_seqs == 0) {
    *empty = true;
    return ATTN_OK;
  }
  if (!out || !q || !k_cache || !v_cache || !block_table || !seq_lens) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned4(block_table) || !aligned4(seq_lens) || !aligned4(lse_out) || !aligned4(status_dev))
    return ATTN_ERR_INVALID_ARG;
  const int64_t pages_needed = ((int64_t)max_seqlen_k + block_size - 1) / block_size;
  if (block_table_stride < 1 || block_table_stride < pages_needed) return ATTN_ERR_INVALID_ARG;
  if (num_seqs > 65535 || (int64_t)num_q_heads > 65535) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

int check_device_sm103() { return check_device(); }

}  // namespace attn

extern "C" {

int32_t attn_abi_version(void) { return 2; }

void attn_tensor_map_cache_stats(uint64_t* hits, uint64_t* misses) {
  if (hits) *hits = attn::g_map_hits.load(std::memory_order_relaxed);
  if (misses) *misses = attn::g_map_misses.load(std::memory_order_relaxed);
}

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case ATTN_ERR_BAD_BLOCK_TABLE: return "block table entry out of range";
    case ATTN_ERR_TIMEOUT: return "pipeline wait timed out";
  }
  return "unknown status";
}

namespace {
// Shared by attn_fwd_prefill and its timeout test hook: the hook passes a
// short wait limit and asks the producer to issue nothing.
attn_status_t prefill_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_table, int32_t block_table_stride,
                           const int32_t* query_start_loc, const int32_t* seq_lens,
                           int32_t num_seqs, int32_t max_seqlen_q, int32_t max_seqlen_k,
                           int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_size, int32_t block_size, int32_t num_blocks, float scale,
                           int32_t causal, attn_dtype_t dtype, attn_round_t rounding,
                           float* lse_out, int32_t* status_dev, void* stream,
                           uint64_t wait_limit_ns, int32_t stall_producer,
                           const attn_features_t* features, bool split = false,
                           void* split_ws = nullptr, size_t split_ws_bytes = 0) {
  // ---- host-side validation (no CUDA call before this block ends)
  Features feat;
  if (read_features(features, feat) != ATTN_OK) return ATTN_ERR_INVALID_ARG;
  if (num_seqs < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || total_q < 0) return ATTN_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (rounding < ATTN_RTNE || rounding > ATTN_OUT_F32) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!valid_scale(scale)) return ATTN_ERR_INVALID_ARG;
  if (block_size <= 0 || num_blocks <= 0) return ATTN_ERR_INVALID_ARG;
  if (head_size != 64 && head_size != 128 && head_size != 256) return ATTN_ERR_UNSUPPORTED;
  if (block_size % 16 != 0 || !(128 % block_size == 0 || block_size % 128 == 0)) return ATTN_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0) return ATTN_OK;  // nothing to compute
  if (!out || !q || !k_cache || !v_cache || !block_table || !query_start_loc || !seq_lens)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned4(block_table) || !aligned4(query_start_loc) || !aligned4(seq_lens) ||
      !aligned4(lse_out) || !aligned4(status_dev))
    return ATTN_ERR_INVALID_ARG;
  const int64_t pages_needed = ((int64_t)max_seqlen_k + block_size - 1) / block_size;
  if (block_table_stride < 1 || block_table_stride < pages_needed) return ATTN_ERR_INVALID_ARG;
  const int group = num_q_heads / num_kv_heads;
  const bool pair_heads = group % 2 == 0;
  const int64_t row_blocks = ((int64_t)max_seqlen_q + 127) / 128;
  int64_t gz = 0, gx = 0;
  prefill_grid(head_size, pair_heads, num_q_heads, row_blocks, gx, gz);
  if (num_seqs > 65535 || gz > 65535 || gx > 2147483647) return ATTN_ERR_UNSUPPORTED;
  if (split && (!split_ws || split_ws_bytes < attn_prefill_split_workspace_size(head_size) ||
                (reinterpret_cast<uintptr_t>(split_ws) & 255u)))
    return ATTN_ERR_WORKSPACE;

  // fp8 caches: the K factor joins tau, the V factor scales the output
  const float scale_eff = feat.kv_fp8 ? scale * feat.k_scale : scale;
  if (!valid_scale(scale_eff)) return ATTN_ERR_INVALID_ARG;
  Fp8Workspace fw;
  if (feat.kv_fp8) {
    if (!fp8_workspace_layout(num_seqs, max_seqlen_k, num_kv_heads, head_size, block_size, fw))
      return ATTN_ERR_INVALID_ARG;
    if (fw.n_pages > 2147483647) return ATTN_ERR_UNSUPPORTED;
    if (!feat.workspace || feat.workspace_bytes < fw.total ||
        (reinterpret_cast<uintptr_t>(feat.workspace) & 255u))
      return ATTN_ERR_WORKSPACE;
  }

  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;

  if (feat.kv_fp8) {
    // widen the referenced pages into the workspace, then run the 16-bit
    // path on that copy through its identity block table
    uint8_t* ws = static_cast<uint8_t*>(feat.workspace);
    void* k16 = ws + fw.k_off;
    void* v16 = ws + fw.v_off;
    int32_t* table = reinterpret_cast<int32_t*>(ws + fw.table_off);
    cudaError_t e = attn::launch_kv_widen(k_cache, v_cache, block_table, block_table_stride,
                                          seq_lens, num_seqs, (int32_t)fw.pages_per_seq,
                                          block_size, num_blocks, fw.page_elems,
                                          dtype == ATTN_BF16, k16, v16, table, status_dev,
                                          static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
    k_cache = k16;
    v_cache = v16;
    block_table = table;
    block_table_stride = (int32_t)fw.pages_per_seq;
    num_blocks = (int32_t)fw.n_pages;
  }

  attn::PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  const bool bf16 = dtype == ATTN_BF16;
  const cuuint64_t d = (cuuint64_t)head_size;
  {
    const cuuint64_t dims[3] = {d, (cuuint64_t)num_q_heads, (cuuint64_t)total_q};
    const cuuint64_t strides[2] = {d * 2, d * 2 * (cuuint64_t)num_q_heads};
    const cuuint32_t box[3] = {64, 1, 128};
    if (!attn::encode_tiled(&p.tm_q, bf16, 3, dims, strides, box, q, CU_TENSOR_MAP_SWIZZLE_128B)) return ATTN_ERR_CUDA;
    // full 128-row output tiles are stored through a map of the same shape
    if (rounding != ATTN_OUT_F32 &&
        !attn::encode_tiled(&p.tm_o, bf16, 3, dims, strides, box, out, CU_TENSOR_MAP_SWIZZLE_128B))
      return ATTN_ERR_CUDA;
  }
  {
    const cuuint64_t dims[4] = {d, (cuuint64_t)num_kv_heads, (cuuint64_t)block_size,
                                (cuuint64_t)num_blocks};
    const cuuint64_t strides[3] = {d * 2, d * 2 * (cuuint64_t)num_kv_heads,
                                   d * 2 * (cuuint64_t)num_kv_heads * (cuuint64_t)block_size};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)(block_size < 128 ? block_size : 128), 1};
    // head size 256 reads V in 64-key halves of a key tile
    const cuuint32_t vbox[4] = {64, 1, (cuuint32_t)(head_size == 256 && block_size > 64 ? 64 : box[2]), 1};
    if (!attn::encode_tiled(&p.tm_k, bf16, 4, dims, strides, box, k_cache, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !attn::encode_tiled(&p.tm_v, bf16, 4, dims, strides, vbox, v_cache, CU_TENSOR_MAP_SWIZZLE_128B))
      return ATTN_ERR_CUDA;
  }
  p.out = out;
  p.lse = lse_out;
  p.status = status_dev;
  p.block_table = block_table;
  p.query_start_loc = query_start_loc;
  p.seq_lens = seq_lens;
  p.bt_stride = block_table_stride;
  p.num_seqs = num_seqs;
  p.max_seqlen_q = max_seqlen_q;
  p.max_seqlen_k = max_seqlen_k;
  p.total_q = total_q;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.box_rows = block_size < 128 ? block_size : 128;
  p.pair_heads = pair_heads ? 1 : 0;
  p.causal = causal;
  p.rounding = (int32_t)rounding;
  p.scale_log2 = scale_eff * kLog2e;
  p.wait_limit_ns = wait_limit_ns;
  p.stall_producer = stall_producer;
  set_features(p, feat, scale_eff);

  // The split grid: head sizes 64 / 128 without feature flags, a batch its
  // tables hold, and more key tiles (at most) than two per SM.
  const bool feat_on = p.win_left >= 0 || p.win_right >= 0 || p.score_xform || p.sinks ||
                       p.out_scale != 1.f;
  if (split && head_size != 256 && !feat_on && !stall_producer && num_seqs <= attn::kSkMaxSeqs &&
      max_seqlen_q <= 65536) {
    const int sms = attn::device_sm_count();
    if (sms <= 0) return ATTN_ERR_CUDA;
    const int64_t key_tiles = ((int64_t)max_seqlen_k + 127) / 128;
    if ((int64_t)num_seqs * gx * gz * key_tiles >= 2 * (int64_t)sms) {
      const int G = sms < attn::kSkMaxCtas ? sms : attn::kSkMaxCtas;
      uint8_t* ws = static_cast<uint8_t*>(split_ws);
      const size_t part_o_bytes = (size_t)2 * attn::kSkMaxCtas * 2 * 128 * (size_t)head_size * 4;
      const size_t part_ml_bytes = (size_t)2 * attn::kSkMaxCtas * 2 * 128 * 2 * 4;
      p.sk_units_x = (int32_t)gx;
      p.sk_part_o = reinterpret_cast<float*>(ws);
      p.sk_part_ml = reinterpret_cast<float*>(ws + part_o_bytes);
      p.sk_ticket = reinterpret_cast<unsigned long long*>(ws + part_o_bytes + part_ml_bytes);
      p.sk_epoch = next_call_epoch();
      cudaError_t e = attn::launch_prefill_streamk(p, head_size, bf16, G, static_cast<cudaStream_t>(stream));
      return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
    }
  }
  dim3 grid((unsigned)gx, (unsigned)num_seqs, (unsigned)gz);
  cudaError_t e = attn::launch_prefill(p, head_size, bf16, grid, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
}  // namespace

size_t attn_prefill_split_workspace_size(int32_t head_size) {
  if (head_size != 64 && head_size != 128 && head_size != 256) return 0;
  const size_t d = head_size == 256 ? 0 : (size_t)head_size;   // 256: the workspace goes unused
  const size_t part_o = (size_t)2 * attn::kSkMaxCtas * 2 * 128 * d * 4;
  const size_t part_ml = (size_t)2 * attn::kSkMaxCtas * 2 * 128 * 2 * 4;
  const size_t tickets = (size_t)attn::kSkMaxCtas * 8;
  return (part_o + part_ml + tickets + 255) / 256 * 256;
}

attn_status_t attn_fwd_prefill_split(void* out, const void* q, const void* k_cache,
                                     const void* v_cache, const int32_t* block_table,
                                     int32_t block_table_stride, const int32_t* query_start_loc,
                                     const int32_t* seq_lens, int32_t num_seqs,
                                     int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t total_q,
                                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                     int32_t block_size, int32_t num_blocks, float scale,
                                     int32_t causal, attn_dtype_t dtype, attn_round_t rounding,
                                     float* lse_out, int32_t* status_dev, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  return prefill_impl(out, q, k_cache, v_cache, block_table, block_table_stride, query_start_loc,
                      seq_lens, num_seqs, max_seqlen_q, max_seqlen_k, total_q, num_q_heads,
                      num_kv_heads, head_size, block_size, num_blocks, scale, causal, dtype,
                      rounding, lse_out, status_dev, stream, kDefaultWaitLimitNs, 0, nullptr, true,
                      workspace, workspace_bytes);
}

attn_status_t attn_fwd_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_table, int32_t block_table_stride,
                               const int32_t* query_start_loc, const int32_t* seq_lens,
                               int32_t num_seqs, int32_t max_seqlen_q, int32_t max_seqlen_k,
                               int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_size, int32_t block_size, int32_t num_blocks,
                               float scale, int32_t causal, attn_dtype_t dtype,
                               attn_round_t rounding, float* lse_out, int32_t* status_dev,
                               void* stream) {
  return prefill_impl(out, q, k_cache, v_cache, block_table, block_table_stride, query_start_loc,
                      seq_lens, num_seqs, max_seqlen_q, max_seqlen_k, total_q, num_q_heads,
                      num_kv_heads, head_size, block_size, num_blocks, scale, causal, dtype,
                      rounding, lse_out, status_dev, stream, kDefaultWaitLimitNs, 0, nullptr);
}

attn_status_t attn_fwd_prefill_ex(void* out, const void* q, const void* k_cache,
                                  const void* v_cache, const int32_t* block_table,
                                  int32_t block_table_stride, const int32_t* query_start_loc,
                                  const int32_t* seq_lens, int32_t num_seqs, int32_t max_seqlen_q,
                                  int32_t max_seqlen_k, int32_t total_q, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                  int32_t num_blocks, float scale, int32_t causal,
                                  attn_dtype_t dtype, attn_round_t rounding, float* lse_out,
                                  int32_t* status_dev, void* stream,
                                  const attn_features_t* features) {
  return prefill_impl(out, q, k_cache, v_cache, block_table, block_table_stride, query_start_loc,
                      seq_lens, num_seqs, max_seqlen_q, max_seqlen_k, total_q, num_q_heads,
                      num_kv_heads, head_size, block_size, num_blocks, scale, causal, dtype,
                      rounding, lse_out, status_dev, stream, kDefaultWaitLimitNs, 0, features);
}

attn_status_t attn_test_prefill_timeout(void* out, const void* q, const void* k_cache,
                                        const void* v_cache, const int32_t* block_table,
                                        int32_t block_table_stride, const int32_t* query_start_loc,
                                        const int32_t* seq_lens, int32_t num_seqs,
                                        int32_t max_seqlen_q, int32_t max_seqlen_k,
                                        int32_t total_q, int32_t num_q_heads,
                                        int32_t num_kv_heads, int32_t head_size,
                                        int32_t block_size, int32_t num_blocks, float scale,
                                        int32_t causal, attn_dtype_t dtype, attn_round_t rounding,
                                        int32_t* status_dev, uint64_t wait_limit_ns, void* stream) {
  if (!status_dev) return ATTN_ERR_INVALID_ARG;
  if (wait_limit_ns < 1000000ull || wait_limit_ns > kDefaultWaitLimitNs) return ATTN_ERR_INVALID_ARG;
  return prefill_impl(out, q, k_cache, v_cache, block_table, block_table_stride, query_start_loc,
                      seq_lens, num_seqs, max_seqlen_q, max_seqlen_k, total_q, num_q_heads,
                      num_kv_heads, head_size, block_size, num_blocks, scale, causal, dtype,
                      rounding, nullptr, status_dev, stream, wait_limit_ns, 1, nullptr);
}

attn_status_t attn_fwd_dense_ex(void* out, const void* q, const void* k, const void* v,
                                const int64_t* q_strides, const int64_t* k_strides,
                                const int64_t* v_strides, const int64_t* o_strides, int32_t batch,
                                int32_t seqlen_q, int32_t seqlen_k, int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t head_size, float scale,
                                int32_t causal, attn_dtype_t dtype, attn_round_t rounding,
                                float* lse_out, int32_t* status_dev, void* stream,
                                const attn_features_t* features) {
  // ---- host-side validation (no CUDA call before this block ends)
  Features feat;
  if (read_features(features, feat) != ATTN_OK) return ATTN_ERR_INVALID_ARG;
  if (batch < 0 || seqlen_q < 0 || seqlen_k < 0) return ATTN_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (rounding < ATTN_RTNE || rounding > ATTN_OUT_F32) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!valid_scale(scale)) return ATTN_ERR_INVALID_ARG;
  if (!q_strides || !k_strides || !v_strides || !o_strides) return ATTN_ERR_INVALID_ARG;
  if (head_size != 64 && head_size != 128 && head_size != 256) return ATTN_ERR_UNSUPPORTED;
  if (batch == 0 || seqlen_q == 0) return ATTN_OK;  // nothing to compute
  if (!out || !q || !k || !v) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k) || !aligned16(v)) return ATTN_ERR_INVALID_ARG;
  if (!aligned4(lse_out) || !aligned4(status_dev)) return ATTN_ERR_INVALID_ARG;
  const int64_t out_elem = rounding == ATTN_OUT_F32 ? 4 : 2;
  const int64_t kv_elem = feat.kv_fp8 ? 1 : 2;     // fp8: one byte per element
  for (int i = 0; i < 3; ++i) {
    // positive strides whose byte sizes are multiples of 16 (TMA and 16-byte stores)
    if (q_strides[i] <= 0 || k_strides[i] <= 0 || v_strides[i] <= 0 || o_strides[i] <= 0) return ATTN_ERR_INVALID_ARG;
    if ((q_strides[i] * 2) % 16 || (k_strides[i] * kv_elem) % 16 || (v_strides[i] * kv_elem) % 16 ||
        (o_strides[i] * out_elem) % 16)
      return ATTN_ERR_INVALID_ARG;
  }
  // fp8: K and V are widened into the workspace (the layout of an fp8
  // prefill over `batch` sequences with one page of seqlen_k rows each)
  const float scale_eff = feat.kv_fp8 ? scale * feat.k_scale : scale;
  if (!valid_scale(scale_eff)) return ATTN_ERR_INVALID_ARG;
  Fp8Workspace fw;
  if (feat.kv_fp8) {
    if (!fp8_workspace_layout(batch, seqlen_k, num_kv_heads, head_size,
                              seqlen_k > 0 ? seqlen_k : 1, fw))
      return ATTN_ERR_INVALID_ARG;
    if (!feat.workspace || feat.workspace_bytes < fw.total ||
        (reinterpret_cast<uintptr_t>(feat.workspace) & 255u))
      return ATTN_ERR_WORKSPACE;
  }
  const int group = num_q_heads / num_kv_heads;
  const bool pair_heads = group % 2 == 0;
  const int64_t row_blocks = ((int64_t)seqlen_q + 127) / 128;
  int64_t gz = 0, gx = 0;
  prefill_grid(head_size, pair_heads, num_q_heads, row_blocks, gx, gz);
  if (batch > 65535 || gz > 65535) return ATTN_ERR_UNSUPPORTED;

  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;

  const bool bf16 = dtype == ATTN_BF16;
  int64_t dense_kv_strides[3];
  if (feat.kv_fp8) {
    uint8_t* ws = static_cast<uint8_t*>(feat.workspace);
    cudaError_t e = attn::launch_kv_widen_dense(k, v, k_strides, v_strides, batch, seqlen_k,
                                                num_kv_heads, head_size, bf16, ws + fw.k_off,
                                                ws + fw.v_off, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
    k = ws + fw.k_off;
    v = ws + fw.v_off;
    dense_kv_strides[0] = (int64_t)seqlen_k * num_kv_heads * head_size;
    dense_kv_strides[1] = (int64_t)num_kv_heads * head_size;
    dense_kv_strides[2] = head_size;
    k_strides = dense_kv_strides;
    v_strides = dense_kv_strides;
  }

  attn::PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  const cuuint64_t d = (cuuint64_t)head_size;
  const cuuint64_t sk_dim = (cuuint64_t)(seqlen_k > 0 ? seqlen_k : 1);   // never read when 0
  {
    // Q and O: dims (d, Hq, Sq, B); the tile box is 128 rows of one head
    const cuuint64_t dims[4] = {d, (cuuint64_t)num_q_heads, (cuuint64_t)seqlen_q, (cuuint64_t)batch};
    const cuuint32_t box[4] = {64, 1, 128, 1};
    const cuuint64_t qs[3] = {(cuuint64_t)q_strides[2] * 2, (cuuint64_t)q_strides[1] * 2, (cuuint64_t)q_strides[0] * 2};
    if (!attn::encode_tiled(&p.tm_q, bf16, 4, dims, qs, box, q, CU_TENSOR_MAP_SWIZZLE_128B)) return ATTN_ERR_CUDA;
    const cuuint64_t os[3] = {(cuuint64_t)o_strides[2] * 2, (cuuint64_t)o_strides[1] * 2, (cuuint64_t)o_strides[0] * 2};
    if (rounding != ATTN_OUT_F32 &&
        !attn::encode_tiled(&p.tm_o, bf16, 4, dims, os, box, out, CU_TENSOR_MAP_SWIZZLE_128B))
      return ATTN_ERR_CUDA;
  }
  {
    // K and V as a paged cache whose page is the batch entry: dims (d, Hkv, Sk, B)
    const cuuint64_t dims[4] = {d, (cuuint64_t)num_kv_heads, sk_dim, (cuuint64_t)batch};
    const cuuint32_t box[4] = {64, 1, 128, 1};
    const cuuint32_t vbox[4] = {64, 1, head_size == 256 ? 64u : 128u, 1};
    const cuuint64_t ks[3] = {(cuuint64_t)k_strides[2] * 2, (cuuint64_t)k_strides[1] * 2, (cuuint64_t)k_strides[0] * 2};
    const cuuint64_t vs[3] = {(cuuint64_t)v_strides[2] * 2, (cuuint64_t)v_strides[1] * 2, (cuuint64_t)v_strides[0] * 2};
    if (!attn::encode_tiled(&p.tm_k, bf16, 4, dims, ks, box, k, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !attn::encode_tiled(&p.tm_v, bf16, 4, dims, vs, vbox, v, CU_TENSOR_MAP_SWIZZLE_128B))
      return ATTN_ERR_CUDA;
  }
  p.out = out;
  p.lse = lse_out;
  p.status = status_dev;
  p.num_seqs = batch;
  p.max_seqlen_q = seqlen_q;
  p.max_seqlen_k = seqlen_k;
  p.total_q = (int32_t)((int64_t)batch * seqlen_q > 2147483647 ? 2147483647 : (int64_t)batch * seqlen_q);
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  // one "page" per batch entry, at least one 128-key box long
  p.block_size = (int32_t)((sk_dim + 127) / 128 * 128);
  p.num_blocks = batch;
  p.box_rows = 128;
  p.pair_heads = pair_heads ? 1 : 0;
  p.dense = 1;
  p.dense_sq = seqlen_q;
  p.dense_sk = seqlen_k;
  p.o_stride_b = o_strides[0];
  p.o_stride_s = o_strides[1];
  p.o_stride_h = o_strides[2];
  p.causal = causal;
  p.rounding = (int32_t)rounding;
  p.scale_log2 = scale_eff * kLog2e;
  p.wait_limit_ns = kDefaultWaitLimitNs;
  set_features(p, feat, scale_eff);

  dim3 grid((unsigned)gx, (unsigned)batch, (unsigned)gz);
  cudaError_t e = attn::launch_prefill(p, head_size, bf16, grid, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_fwd_dense(void* out, const void* q, const void* k, const void* v,
                             const int64_t* q_strides, const int64_t* k_strides,
                             const int64_t* v_strides, const int64_t* o_strides, int32_t batch,
                             int32_t seqlen_q, int32_t seqlen_k, int32_t num_q_heads,
                             int32_t num_kv_heads, int32_t head_size, float scale, int32_t causal,
                             attn_dtype_t dtype, attn_round_t rounding, float* lse_out,
                             int32_t* status_dev, void* stream) {
  return attn_fwd_dense_ex(out, q, k, v, q_strides, k_strides, v_strides, o_strides, batch,
                           seqlen_q, seqlen_k, num_q_heads, num_kv_heads, head_size, scale, causal,
                           dtype, rounding, lse_out, status_dev, stream, nullptr);
}

size_t attn_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t head_size,
                                  int32_t num_splits) {
  if (num_seqs <= 0 || num_q_heads <= 0 || head_size <= 0 || num_splits <= 0) return 0;
  const size_t counter_bytes = 256;
  if (num_splits == 1) return counter_bytes;
  const size_t rows = (size_t)num_seqs * (size_t)num_q_heads * (size_t)num_splits;
  return rows * (size_t)head_size * sizeof(float) + rows * 2 * sizeof(float) + counter_bytes;
}

size_t attn_fp8_prefill_workspace_size(int32_t num_seqs, int32_t max_seqlen_k,
                                       int32_t num_kv_heads, int32_t head_size,
                                       int32_t block_size) {
  Fp8Workspace w;
  if (!fp8_workspace_layout(num_seqs, max_seqlen_k, num_kv_heads, head_size, block_size, w)) return 0;
  return w.total;
}

attn_status_t attn_fwd_decode_ex(void* out, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* block_table,
                                 int32_t block_table_stride, const int32_t* seq_lens,
                                 int32_t num_seqs, int32_t max_seqlen_k, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                 int32_t num_blocks, float scale, int32_t num_splits,
                                 attn_dtype_t dtype, attn_round_t rounding, float* lse_out,
                                 void* workspace, size_t workspace_bytes, int32_t* status_dev,
                                 void* stream, const attn_features_t* features) {
  Features feat;
  if (read_features(features, feat) != ATTN_OK) return ATTN_ERR_INVALID_ARG;
  bool empty = false;
  const int chk = attn::check_decode_args(out, q, k_cache, v_cache, block_table, block_table_stride,
                                          seq_lens, num_seqs, max_seqlen_k, num_q_heads,
                                          num_kv_heads, head_size, block_size, num_blocks, scale,
                                          num_splits, (int)dtype, (int)rounding, lse_out,
                                          status_dev, &empty);
  if (chk != ATTN_OK || empty) return (attn_status_t)chk;
  const size_t need = attn_decode_workspace_size(num_seqs, num_q_heads, head_size, num_splits);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;

  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;

  attn::DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.out = out;
  p.lse = lse_out;
  p.status = status_dev;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.bt_stride = block_table_stride;
  p.num_seqs = num_seqs;
  p.max_seqlen_k = max_seqlen_k;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.num_splits = num_splits;
  p.rounding = (int32_t)rounding;
  // fp8 caches: the K factor joins tau, the V factor scales the output
  const float scale_eff = feat.kv_fp8 ? scale * feat.k_scale : scale;
  if (!valid_scale(scale_eff)) return ATTN_ERR_INVALID_ARG;
  p.scale_log2 = scale_eff * kLog2e;
  p.scale = scale_eff;
  p.kv_fp8 = feat.kv_fp8 ? 1 : 0;
  p.out_scale = feat.kv_fp8 ? feat.v_scale : 1.f;
  p.win_left = feat.win_left;      // the right bound never cuts a decode row (diag = kv_len - 1)
  p.softcap = feat.softcap;
  p.alibi = feat.alibi;
  p.sinks = feat.sinks;
  p.score_xform = (feat.softcap > 0.f || feat.alibi) ? 1 : 0;
  return (attn_status_t)attn::decode_prepare_and_launch(p, head_size, dtype == ATTN_BF16, workspace,
                                                        static_cast<cudaStream_t>(stream));
}

attn_status_t attn_fwd_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_table, int32_t block_table_stride,
                              const int32_t* seq_lens, int32_t num_seqs, int32_t max_seqlen_k,
                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                              int32_t block_size, int32_t num_blocks, float scale,
                              int32_t num_splits, attn_dtype_t dtype, attn_round_t rounding,
                              float* lse_out, void* workspace, size_t workspace_bytes,
                              int32_t* status_dev, void* stream) {
  return attn_fwd_decode_ex(out, q, k_cache, v_cache, block_table, block_table_stride, seq_lens,
                            num_seqs, max_seqlen_k, num_q_heads, num_kv_heads, head_size,
                            block_size, num_blocks, scale, num_splits, dtype, rounding, lse_out,
                            workspace, workspace_bytes, status_dev, stream, nullptr);
}

attn_status_t attn_round_f32(void* out, const float* in, int64_t n, attn_dtype_t dtype,
                             attn_round_t rounding, void* stream) {
  if (n < 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (rounding < ATTN_RTNE || rounding > ATTN_RTZ) return ATTN_ERR_INVALID_ARG;
  if (n == 0) return ATTN_OK;
  if (!out || !in) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(out) & 1u) || !aligned4(in)) return ATTN_ERR_INVALID_ARG;
  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;
  cudaError_t e = attn::launch_round(out, in, n, dtype == ATTN_BF16, (int)rounding,
                                     static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"

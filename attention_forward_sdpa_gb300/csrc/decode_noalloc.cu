// decode_noalloc.cu -- attn_fwd_decode_noalloc: the split-KV decode for
// callers that cannot allocate device memory at all.
//
// Who needs it: callers that are not allowed to allocate device memory.
// A latency-critical serving loop cannot afford cudaMalloc there: it may
// synchronise the device and its cost is unbounded.  A host framework whose
// allocator owns all device memory, or a plugin interface that hands a
// library only its input and output pointers, gives the library no way to
// obtain a workspace.  attn_fwd_decode needs a caller-provided workspace for
// the per-split partial results; this variant keeps that scratch in a fixed
// device array that lives in the library itself.
//
// The array is a file-scope __device__ object, so every GPU that loads the
// library holds ATTN_DECODE_NOALLOC_SCRATCH_BYTES of it until the process
// exits.  Host code cannot use the array's name as a device address: the
// first call on each device looks the address up with cudaGetSymbolAddress
// (with that device current) and caches it.  That first call may load the
// module, so make it before any stream capture.
//
// Every call on a device shares the one array.  Each call first zeroes the
// work counter at the end of its part of the array (the only value that must
// start at zero) and then overwrites every partial o, m and l before the
// combine reads it, so nothing of a previous call is read.  Calls that can
// overlap on the device -- different streams without ordering between them --
// race on the array and must not be issued.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/attn_fwd.h"
#include "attn_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// the scratch: ATTN_DECODE_NOALLOC_SCRATCH_BYTES bytes, 256-byte aligned
static __device__ __align__(256) unsigned char g_decode_scratch[ATTN_DECODE_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" attn_status_t attn_fwd_decode_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
    int32_t block_table_stride, const int32_t* seq_lens, int32_t num_seqs, int32_t max_seqlen_k,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size, int32_t block_size,
    int32_t num_blocks, float scale, int32_t num_splits, attn_dtype_t dtype, attn_round_t rounding,
    float* lse_out, int32_t* status_dev, void* stream) {
  // the same argument rules as attn_fwd_decode
  if (num_seqs < 0 || max_seqlen_k < 0) return ATTN_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (rounding < ATTN_RTNE || rounding > ATTN_OUT_F32) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (block_size <= 0 || num_blocks <= 0) return ATTN_ERR_INVALID_ARG;
  if (num_splits < 1 || num_splits > 64) return ATTN_ERR_INVALID_ARG;
  if (head_size != 64 && head_size != 128 && head_size != 256) return ATTN_ERR_UNSUPPORTED;
  if (block_size % 16 != 0) return ATTN_ERR_UNSUPPORTED;
  if (num_seqs == 0) return ATTN_OK;
  if (!out || !q || !k_cache || !v_cache || !block_table || !seq_lens) return ATTN_ERR_INVALID_ARG;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(q) |
                        reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache);
  if (mis & 15u) return ATTN_ERR_INVALID_ARG;
  const uintptr_t mis4 = reinterpret_cast<uintptr_t>(block_table) |
                         reinterpret_cast<uintptr_t>(seq_lens) |
                         reinterpret_cast<uintptr_t>(lse_out) |
                         reinterpret_cast<uintptr_t>(status_dev);
  if (mis4 & 3u) return ATTN_ERR_INVALID_ARG;
  const int64_t pages_needed = ((int64_t)max_seqlen_k + block_size - 1) / block_size;
  if (block_table_stride < 1 || block_table_stride < pages_needed) return ATTN_ERR_INVALID_ARG;
  if (num_seqs > 65535 || num_q_heads > 65535) return ATTN_ERR_UNSUPPORTED;
  // the problem must fit the built-in scratch
  const size_t need = attn_decode_workspace_size(num_seqs, num_q_heads, head_size, num_splits);
  if (need > (size_t)ATTN_DECODE_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_WORKSPACE;

  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (major != 10 || minor != 3) return ATTN_ERR_UNSUPPORTED;

  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return ATTN_ERR_CUDA;

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
  p.scale_log2 = scale * 1.4426950408889634f;
  p.scale = scale;
  p.win_left = -1;   // no feature flags on this entry point
  p.out_scale = 1.f;
  return (attn_status_t)attn::decode_prepare_and_launch(p, head_size, dtype == ATTN_BF16, scratch,
                                                        static_cast<cudaStream_t>(stream));
}

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
// exits.  Host code cannot use the array's name as a device address: every
// call looks the address up with cudaGetSymbolAddress, with the caller's
// device current, and passes it to the kernels.  The lookup is cheap once
// the library's device code is loaded in that context, and a fresh lookup
// stays right after a device reset or in another context, where the array
// lives at another address.  The first call in a context may load the
// module, so make it before any stream capture.
//
// Every call on a device shares the one array.  The tcgen05 decode path
// zeroes its work counter (in the array, after the partials) on the stream
// before its launch; the SIMT path does not use the counter.  Both write
// every partial o, m and l before the combine reads it, so nothing a
// previous call left in the array is read.  Calls that can overlap on the
// device -- different streams without ordering between them -- race on the
// array and must not be issued.

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/attn_fwd.h"
#include "attn_internal.h"

namespace {

// the scratch: ATTN_DECODE_NOALLOC_SCRATCH_BYTES bytes, 256-byte aligned
static __device__ __align__(256) unsigned char g_decode_scratch[ATTN_DECODE_NOALLOC_SCRATCH_BYTES];

}  // namespace

extern "C" attn_status_t attn_fwd_decode_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
    int32_t block_table_stride, const int32_t* seq_lens, int32_t num_seqs, int32_t max_seqlen_k,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size, int32_t block_size,
    int32_t num_blocks, float scale, int32_t num_splits, attn_dtype_t dtype, attn_round_t rounding,
    float* lse_out, int32_t* status_dev, void* stream) {
  // the same argument rules as attn_fwd_decode
  bool empty = false;
  const int chk = attn::check_decode_args(out, q, k_cache, v_cache, block_table, block_table_stride,
                                          seq_lens, num_seqs, max_seqlen_k, num_q_heads,
                                          num_kv_heads, head_size, block_size, num_blocks, scale,
                                          num_splits, (int)dtype, (int)rounding, lse_out,
                                          status_dev, &empty);
  if (chk != ATTN_OK || empty) return (attn_status_t)chk;
  // the problem must fit the built-in scratch
  const size_t need = attn_decode_workspace_size(num_seqs, num_q_heads, head_size, num_splits);
  if (need > (size_t)ATTN_DECODE_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_WORKSPACE;
  const int dev_ok = attn::check_device_sm103();
  if (dev_ok != ATTN_OK) return (attn_status_t)dev_ok;

  // the array's address in the current context (see the top of the file)
  void* scratch = nullptr;
  if (cudaGetSymbolAddress(&scratch, g_decode_scratch) != cudaSuccess || !scratch)
    return ATTN_ERR_CUDA;

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

// attn_internal.h -- parameter blocks shared by the C-ABI layer and the
// kernel launchers (not part of the public interface).
#pragma once

#include <atomic>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace attn {

// One prefill launch.  Tensor maps are encoded on the host (attn_api.cu).
struct PrefillParams {
  CUtensorMap tm_q;   // Q  [total_q, Hq, d]: dims (d, Hq, total_q), box (64, 1, 128), 128B swizzle;
                      //    dense: dims (d, Hq, Sq, B), box (64, 1, 128, 1)
  CUtensorMap tm_k;   // K  [num_blocks, bs, Hkv, d]: dims (d, Hkv, bs, num_blocks), box (64, 1, R, 1)
  CUtensorMap tm_v;   // V  same as K; head size 256: box rows min(block_size, 64)
  CUtensorMap tm_o;   // O  like Q over the output (16-bit output only): 3-D packed, 4-D dense
  void* out;          // [total_q, Hq, d] 16-bit, or fp32 when rounding == 3
  float* lse;         // [total_q, Hq] or nullptr
  int32_t* status;    // device status word or nullptr
  const int32_t* block_table;
  const int32_t* query_start_loc;
  const int32_t* seq_lens;
  int32_t bt_stride;
  int32_t num_seqs;
  int32_t max_seqlen_q;
  int32_t max_seqlen_k;
  int32_t total_q;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t block_size;
  int32_t num_blocks;
  int32_t box_rows;     // rows of one K/V TMA box = min(block_size, 128)
  int32_t pair_heads;   // 1: the two Q tiles of a CTA are two heads of one group
  int32_t dense;        // 1: fixed-length strided batch (no block table, page = batch index)
  int32_t dense_sq;     // dense: query length of every sequence
  int32_t dense_sk;     // dense: kv length of every sequence
  int64_t o_stride_b;   // dense: output element strides (batch, row, head)
  int64_t o_stride_s;
  int64_t o_stride_h;
  int32_t causal;
  int32_t rounding;     // 0 RTNE, 1 RTNA, 2 RTZ, 3 fp32 output
  float scale_log2;     // tau * log2(e)
  uint64_t wait_limit_ns;  // limit of every pipeline wait (the library default, or a test's)
  int32_t stall_producer;  // test only: the producer issues no copy, so the first wait runs out
  // feature flags (attn_features_t): window bounds (-1 unbounded), softcap
  // (0 off), per-head ALiBi slopes and sink logits (device, or nullptr)
  int32_t win_left;
  int32_t win_right;
  int32_t score_xform;  // 1 when softcap or ALiBi rewrite the scores
  float softcap;
  float scale;          // tau, for the score rewrite
  const float* alibi;
  const float* sinks;
  float out_scale;      // factor on the normalised output (fp8 V factor; 1 otherwise)
  // persistent stream-K launch (prefill_streamk.cu): head units per sequence,
  // the workspace's partial results and tickets, and the call's epoch
  int32_t sk_units_x;
  float* sk_part_o;               // [2 G][2 tiles][128 rows][d] un-normalised o of unit parts
  float* sk_part_ml;              // [2 G][2 tiles][128 rows][2] (m in log2 units, l)
  unsigned long long* sk_ticket;  // [G] (epoch << 16 | parts counted)
  uint64_t sk_epoch;
};

// Largest grid and batch the persistent stream-K prefill takes (its
// workspace holds 2 parts per CTA; its shared-memory tables one entry per
// sequence).
constexpr int kSkMaxCtas = 160;
constexpr int kSkMaxSeqs = 256;

struct DecodeParams {
  CUtensorMap tm_q;     // Q [num_seqs, Hq, d]: dims (d, Hq, num_seqs), box (64, min(16, Hq), 1)
  CUtensorMap tm_k;     // K cache: dims (d, bs, Hkv, num_blocks), box (64, 16, F, 1)
  CUtensorMap tm_v;     // V cache: dims (64, bs, 2, Hkv, num_blocks), box (64, 16, 2, F, 1)
  int32_t* counter;     // work counter of the persistent kernel (zeroed before the launch)
  int32_t n_items;      // num_seqs * (Hq / heads_per_item) * num_splits
  int32_t heads_per_item;  // query heads per KV head in a work item
  int32_t kv_per_item;     // KV heads per work item
  int32_t q_box_rows;
  const void* q;        // [num_seqs, Hq, d]
  const void* k_cache;  // [num_blocks, bs, Hkv, d]
  const void* v_cache;  // [num_blocks, bs, Hkv, d]
  void* out;            // [num_seqs, Hq, d] 16-bit, or fp32 when rounding == 3
  float* lse;           // [num_seqs, Hq] or nullptr
  int32_t* status;
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* part_o;        // [num_seqs, Hq, splits, d] un-normalised partial outputs
  float* part_ml;       // [num_seqs, Hq, splits, 2] (running max in log2 units, denominator)
  int32_t bt_stride;
  int32_t num_seqs;
  int32_t max_seqlen_k;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t block_size;
  int32_t num_blocks;
  int32_t num_splits;
  int32_t rounding;
  float scale_log2;
  // feature flags, as in PrefillParams (both split kernels and the merge
  // honour them)
  int32_t win_left;
  int32_t score_xform;
  float softcap;
  float scale;
  const float* alibi;
  const float* sinks;
  // fp8 caches: K/V hold E4M3 codes; the K factor is folded into scale and
  // scale_log2, the V factor is out_scale (applied to the normalised output)
  int32_t kv_fp8;
  float out_scale;
};

// Launchers return a cudaError_t from the launch.
cudaError_t launch_prefill(const PrefillParams& p, int head_size, bool bf16, dim3 grid,
                           cudaStream_t stream);
cudaError_t launch_prefill_d256(const PrefillParams& p, bool bf16, dim3 grid, cudaStream_t stream);
// The persistent stream-K prefill (head sizes 64 and 128, no feature flags):
// `grid` CTAs, at most kSkMaxCtas.
cudaError_t launch_prefill_streamk(const PrefillParams& p, int head_size, bool bf16, int grid,
                                   cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, int head_size, bool bf16, int group,
                          cudaStream_t stream);
cudaError_t launch_decode_tc(const DecodeParams& p, int head_size, bool bf16, int grid,
                             cudaStream_t stream);
cudaError_t launch_decode_combine(const DecodeParams& p, int head_size, bool bf16,
                                  cudaStream_t stream);

// Shared by the two decode entry points: fills the kernel parameters from
// the (already validated) arguments, places the partials and the work
// counter in `workspace` (attn_decode_workspace_size bytes), and launches.
// Returns an attn_status_t value.
int decode_prepare_and_launch(DecodeParams& p, int head_size, bool bf16, void* workspace,
                              cudaStream_t stream);

// The argument rules the decode entry points share: everything except the
// workspace and the device check, in one place so that the entry points
// accept the same inputs.  Returns an attn_status_t value; ATTN_OK with
// *empty set means there is nothing to launch (num_seqs == 0).
int check_decode_args(const void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_table, int32_t block_table_stride,
                      const int32_t* seq_lens, int32_t num_seqs, int32_t max_seqlen_k,
                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                      int32_t block_size, int32_t num_blocks, float scale, int32_t num_splits,
                      int dtype, int rounding, const float* lse_out, const int32_t* status_dev,
                      bool* empty);

// ATTN_OK when the current device is an sm_103 GPU (the only target the
// kernels are built for), else ATTN_ERR_UNSUPPORTED or ATTN_ERR_CUDA.
int check_device_sm103();

bool encode_tiled(CUtensorMap* map, bool bf16, int rank, const cuuint64_t* dims,
                  const cuuint64_t* strides_bytes, const cuuint32_t* box, const void* base,
                  CUtensorMapSwizzle swz);
// The same for a tensor of bytes (fp8 codes).
bool encode_tiled_u8(CUtensorMap* map, int rank, const cuuint64_t* dims,
                     const cuuint64_t* strides_bytes, const cuuint32_t* box, const void* base,
                     CUtensorMapSwizzle swz);
int device_sm_count();

// Opts `kernel` in to `bytes` of dynamic shared memory on the current device.
// Function attributes are per device, so `done` (one per kernel) records the
// devices already set up; setting an attribute twice is harmless, so two
// threads racing here only repeat the call.
template <typename Kernel>
cudaError_t ensure_dynamic_smem(Kernel kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
  return e;
}

cudaError_t launch_round(void* out, const float* in, int64_t n, bool bf16, int mode,
                         cudaStream_t stream);

// fp8 prefill: widens the pages that each sequence references (E4M3 codes ->
// exact 16-bit values) into a dense page array, page (b, p) at index
// b * pages_per_seq + p, and writes the matching identity block table
// [num_seqs, pages_per_seq].  A referenced page id outside [0, num_blocks)
// is reported on the status word and its copy is zero.
cudaError_t launch_kv_widen(const void* k8, const void* v8, const int32_t* block_table,
                            int32_t bt_stride, const int32_t* seq_lens, int32_t num_seqs,
                            int32_t pages_per_seq, int32_t block_size, int32_t num_blocks,
                            int64_t page_elems, bool bf16, void* k16, void* v16,
                            int32_t* table_out, int32_t* status, cudaStream_t stream);

// fp8 dense: widens logical [B, Sk, Hkv, d] E4M3 K and V with the given
// (batch, row, head) strides (in bytes, channels contiguous) into contiguous
// 16-bit [B, Sk, Hkv, d] copies.
cudaError_t launch_kv_widen_dense(const void* k8, const void* v8, const int64_t* k_strides,
                                  const int64_t* v_strides, int32_t batch, int32_t seqlen_k,
                                  int32_t num_kv_heads, int32_t head_size, bool bf16, void* k16,
                                  void* v16, cudaStream_t stream);

// In-kernel error codes written to the status word (same values as the
// public attn_status_t).
enum : int32_t { kStatusBadArg = 1, kStatusBadBlockTable = 5, kStatusTimeout = 6 };

__device__ __forceinline__ void report_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

}  // namespace attn

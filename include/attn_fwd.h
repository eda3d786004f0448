/*
 * attn_fwd.h -- C ABI of the GB300 (sm_103a) fused scaled-dot-product-attention
 * forward library (libattn_fwd_sm103.so).
 *
 * What it computes.  For every sequence b, query head h and query row i:
 *     O[i, h, :] = sum_j softmax_j(tau * <Q[i, h, :], K[j, kvh, :]>) V[j, kvh, :]
 * over the visible keys j, with kvh = h / (num_q_heads / num_kv_heads).  This
 * is the specification of "gfx942 unified attention, from the math up",
 * sec. 1, evaluated by the online-softmax recurrence of sec. 3 (running max m,
 * denominator l, rescale alpha = e^(m_old - m_new), un-normalised o, final
 * o / l) without ever forming the query-by-key score matrix.  Keys are read
 * from a paged cache through a block table (sec. 5); GQA groups follow the
 * repeat_interleave convention of sec. 5 and sec. 10.  Causal masking is
 * bottom-right aligned (sec. 4, and the "Troubleshooting" section of
 * "gfx942 unified attention - parity + benchmark harness"): row i of a
 * sequence with query length Sq and kv length Sk sees keys j <= i + Sk - Sq.
 * A row that sees no key (causal with Sq > Sk, or Sk = 0) gets O = 0 and
 * log-sum-exp -inf.  Output rounding modes are those of "MoonMath.ai abre un
 * nucleo de atencion HIP para AMD MI300X ..." (7minutos.es), section "Punto de
 * referencia": RTNE, RTNA (ties away from zero) and RTZ.
 *
 * Memory and threading rules for every entry point:
 *   - Every pointer argument is caller-owned DEVICE memory unless stated
 *     otherwise; tensors are dense, row-major, with the shapes given.  The
 *     library never allocates or frees device memory and keeps no pointer
 *     after the call returns.
 *   - Alignment: tensors of 16-bit elements and workspaces as stated at each
 *     entry point (16 bytes or more); int32 and fp32 arrays (block tables,
 *     query_start_loc, seq_lens, lse_out, status_dev, the fp32 input of
 *     attn_round_f32) on 4 bytes; the output of attn_round_f32 on 2.  A
 *     misaligned pointer is ATTN_ERR_INVALID_ARG (a misaligned workspace
 *     ATTN_ERR_WORKSPACE).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  Inputs must stay valid until the work completes.
 *   - Argument errors are detected on the host and returned before anything
 *     is launched.  A failed launch returns ATTN_ERR_CUDA.  Errors that can
 *     only be seen on the device (a block-table entry outside [0, num_blocks),
 *     a sequence longer than max_seqlen_*, a wait that timed out) are written
 *     to *status_dev when it is non-NULL (first error wins; the caller sets it
 *     to 0 beforehand and reads it after synchronising); the offending work is
 *     skipped or loads zeros, never reads outside the given tensors.
 *   - Nothing throws across the ABI.  The library requires a compute
 *     capability 10.3 (sm_103) device; otherwise ATTN_ERR_UNSUPPORTED.
 */
#ifndef ATTN_FWD_H_
#define ATTN_FWD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,   /* bad pointer, size or enum value */
  ATTN_ERR_UNSUPPORTED = 2,   /* valid request outside the compiled set */
  ATTN_ERR_CUDA = 3,          /* a CUDA call or launch failed */
  ATTN_ERR_WORKSPACE = 4,     /* workspace missing, too small or misaligned */
  ATTN_ERR_BAD_BLOCK_TABLE = 5, /* (device status only) page id out of range */
  ATTN_ERR_TIMEOUT = 6        /* (device status only) a pipeline wait timed out */
} attn_status_t;

typedef enum { ATTN_F16 = 0, ATTN_BF16 = 1 } attn_dtype_t;

/* Output rounding: RTNE = nearest, ties to even; RTNA = nearest, ties away
 * from zero; RTZ = toward zero.  ATTN_OUT_F32 writes the fp32 value o / l
 * unrounded (out is then float*). */
typedef enum { ATTN_RTNE = 0, ATTN_RTNA = 1, ATTN_RTZ = 2, ATTN_OUT_F32 = 3 } attn_round_t;

/*
 * attn_fwd_prefill -- prefill / dense forward over packed queries and a paged
 * KV cache ("gfx942 unified attention, from the math up", sec. 3-5).
 *
 *   out          [total_q, num_q_heads, head_size], dtype (fp32 for ATTN_OUT_F32)
 *   q            [total_q, num_q_heads, head_size], dtype; 16-byte aligned
 *   k_cache      [num_blocks, block_size, num_kv_heads, head_size], dtype; 16-byte aligned
 *   v_cache      same shape as k_cache
 *   block_table  [num_seqs, block_table_stride] int32: page ids of each
 *                sequence's keys in order (key j of sequence b lives in page
 *                block_table[b][j / block_size], slot j % block_size); only
 *                the first ceil(seq_lens[b] / block_size) entries are read.
 *   query_start_loc [num_seqs + 1] int32: prefix sum of query lengths;
 *                sequence b owns rows [query_start_loc[b], query_start_loc[b+1]).
 *   seq_lens     [num_seqs] int32: kv length of each sequence.
 *   max_seqlen_q / max_seqlen_k: upper bounds of the per-sequence lengths
 *                (used to size the grid; violations are reported on the device).
 *   head_size    64, 128 or 256 (the pages leave 256 without a tiled kernel,
 *                "gfx942 unified attention -- parity + benchmark harness",
 *                Troubleshooting; here it has one).  block_size: a multiple of 16 that divides 128,
 *                or a multiple of 128.  num_q_heads % num_kv_heads == 0.
 *   scale        tau (> 0), normally 1/sqrt(head_size).
 *   causal       0 or 1 (bottom-right aligned).
 *   lse_out      optional [total_q, num_q_heads] fp32 natural-log log-sum-exp
 *                of each row's scaled scores, or NULL.
 *   status_dev   optional device int32 status word, or NULL.
 *   stream       cudaStream_t.
 * Dense BSHD input [B, S, H, d] is the special case query_start_loc =
 * {0, S, 2S, ...}, block_size = S, num_blocks = B, block_table[b] = {b}.
 */
attn_status_t attn_fwd_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_table, int32_t block_table_stride,
                               const int32_t* query_start_loc, const int32_t* seq_lens,
                               int32_t num_seqs, int32_t max_seqlen_q, int32_t max_seqlen_k,
                               int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_size, int32_t block_size, int32_t num_blocks,
                               float scale, int32_t causal, attn_dtype_t dtype,
                               attn_round_t rounding, float* lse_out, int32_t* status_dev,
                               void* stream);

/*
 * attn_fwd_prefill_split -- attn_fwd_prefill with the key range of work units
 * split across a persistent grid, so that every SM gets the same number of
 * key tiles whatever the row lengths: the tail KV split for the fractional
 * last wave of MoonMath's HIP kernel (7minutos.es, "Dónde viven los datos y
 * por qué 16x16x16"), with the parts of a split unit merged by the
 * log-sum-exp combine of "gfx942 unified attention, from the math up",
 * sec. 8.  A unit is two 128-row query tiles sharing a KV head; all key
 * tiles of all units are laid end to end and cut into equal ranges, one per
 * CTA; the CTA that finishes the last part of a cut unit merges its parts
 * in key order.
 *
 *   arguments    as attn_fwd_prefill, plus:
 *   workspace    device memory of at least
 *                attn_prefill_split_workspace_size(head_size) bytes,
 *                256-byte aligned, owned by the caller.  It needs no
 *                initialisation and keeps nothing between calls that a
 *                later call reads (each call tags its merge tickets with a
 *                fresh call number), but calls that may run at the same
 *                time must not share it.
 * Results match attn_fwd_prefill within the same tolerance but are not
 * bit-identical to it (a merged unit sums its keys in two or three parts);
 * they are bit-identical from run to run (the merge order is fixed).  Head
 * sizes 64 and 128 with at most 256 sequences take the split grid; other
 * calls, and problems too small to fill the GPU, run attn_fwd_prefill's
 * kernel and leave the workspace untouched.  Errors: as attn_fwd_prefill; a
 * missing, short or misaligned workspace gives ATTN_ERR_WORKSPACE.
 */
size_t attn_prefill_split_workspace_size(int32_t head_size);
attn_status_t attn_fwd_prefill_split(void* out, const void* q, const void* k_cache,
                                     const void* v_cache, const int32_t* block_table,
                                     int32_t block_table_stride, const int32_t* query_start_loc,
                                     const int32_t* seq_lens, int32_t num_seqs,
                                     int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t total_q,
                                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                     int32_t block_size, int32_t num_blocks, float scale,
                                     int32_t causal, attn_dtype_t dtype, attn_round_t rounding,
                                     float* lse_out, int32_t* status_dev, void* workspace,
                                     size_t workspace_bytes, void* stream);

/*
 * attn_fwd_dense -- the same forward for fixed-length batches held as strided
 * tensors, with no block table: logical shapes Q, O [batch, seqlen_q,
 * num_q_heads, head_size] and K, V [batch, seqlen_k, num_kv_heads, head_size]
 * in any (batch, sequence, head) stride order, so that both the BSHD and the
 * BHSD layouts of "MoonMath.ai abre un nucleo de atencion HIP para AMD MI300X
 * ..." (7minutos.es), section "Entendiendo el nucleo", are read in place.
 *
 *   out, q, k, v element (b, i, h, c) lives at base + b*strides[0] + i*strides[1]
 *                + h*strides[2] + c (c = channel, contiguous).  BSHD
 *                [B, S, H, d]: strides {S*H*d, H*d, d}; BHSD [B, H, S, d]:
 *                strides {H*S*d, d, S*d}.  out is dtype (fp32 for
 *                ATTN_OUT_F32), the others dtype; base pointers 16-byte
 *                aligned and every stride a multiple of 16 bytes.
 *   q_strides, k_strides, v_strides, o_strides: HOST arrays of 3 int64 element
 *                strides {batch, sequence, head}; read during the call only.
 *   batch, seqlen_q, seqlen_k, num_q_heads, num_kv_heads, head_size (64, 128 or 256),
 *   scale, causal (bottom-right aligned), dtype, rounding: as for attn_fwd_prefill.
 *   lse_out      optional [batch, num_q_heads, seqlen_q] fp32, or NULL.
 *   status_dev, stream: as for attn_fwd_prefill.
 * The arithmetic is that of attn_fwd_prefill on the equivalent packed and
 * paged tensors (block_size = seqlen_k, block_table[b] = {b}); the results
 * are bit-identical to it.
 */
attn_status_t attn_fwd_dense(void* out, const void* q, const void* k, const void* v,
                             const int64_t* q_strides, const int64_t* k_strides,
                             const int64_t* v_strides, const int64_t* o_strides, int32_t batch,
                             int32_t seqlen_q, int32_t seqlen_k, int32_t num_q_heads,
                             int32_t num_kv_heads, int32_t head_size, float scale, int32_t causal,
                             attn_dtype_t dtype, attn_round_t rounding, float* lse_out,
                             int32_t* status_dev, void* stream);

/*
 * attn_test_prefill_timeout -- TEST HOOK for the failure path, not for
 * production use; the pages have no counterpart.  Launches attn_fwd_prefill's
 * kernel with every pipeline wait limited to wait_limit_ns (1 ms .. 4 s;
 * attn_fwd_prefill uses 4 s) and a producer that issues no copy, so that the
 * first wait of every CTA runs out.  Each CTA then raises its abort flag,
 * releases its tensor memory and records ATTN_ERR_TIMEOUT in *status_dev
 * (required here, caller-zeroed); nothing is written to out, no copy or
 * product is left in flight, and the device stays usable for the next call.
 * Other arguments as attn_fwd_prefill (no lse).  Returns ATTN_OK when the
 * launch succeeded; the timeout itself is reported through *status_dev.
 */
attn_status_t attn_test_prefill_timeout(void* out, const void* q, const void* k_cache,
                                        const void* v_cache, const int32_t* block_table,
                                        int32_t block_table_stride, const int32_t* query_start_loc,
                                        const int32_t* seq_lens, int32_t num_seqs,
                                        int32_t max_seqlen_q, int32_t max_seqlen_k,
                                        int32_t total_q, int32_t num_q_heads,
                                        int32_t num_kv_heads, int32_t head_size,
                                        int32_t block_size, int32_t num_blocks, float scale,
                                        int32_t causal, attn_dtype_t dtype, attn_round_t rounding,
                                        int32_t* status_dev, uint64_t wait_limit_ns, void* stream);

/*
 * attn_decode_workspace_size -- bytes of device workspace attn_fwd_decode
 * needs for these sizes: the split partials (num_seqs * num_q_heads *
 * num_splits * (head_size + 2) fp32 values when num_splits > 1) plus 256
 * bytes for the work counter of the persistent decode kernel.  Pure host
 * arithmetic; 0 only for an empty problem.
 */
size_t attn_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t head_size,
                                  int32_t num_splits);

/*
 * attn_fwd_decode -- one query row per sequence attending to all of its
 * kv_len keys (decode: causal and non-causal coincide for a single query,
 * "gfx942 unified attention, from the math up", sec. 4), by the split-KV
 * scheme of sec. 8: the keys of each sequence are cut into num_splits
 * contiguous parts of ceil(ceil(kv_len / num_splits) / 16) * 16 keys, each
 * part reduced to a partial softmax state in the workspace, and the parts
 * merged by the log-sum-exp rule.
 *
 *   out          [num_seqs, num_q_heads, head_size], dtype (fp32 for ATTN_OUT_F32)
 *   q            [num_seqs, num_q_heads, head_size], dtype
 *   k_cache, v_cache, block_table, block_table_stride, seq_lens,
 *   num_q_heads, num_kv_heads, head_size, block_size, num_blocks, scale:
 *                as for attn_fwd_prefill, except that block_size only needs
 *                to be a multiple of 16.
 *   num_splits   1 .. 64.
 *   lse_out      optional [num_seqs, num_q_heads] fp32, or NULL.
 *   workspace    device memory of at least attn_decode_workspace_size(...)
 *                bytes, 16-byte aligned; owned by the caller, any initial
 *                contents (the call zeroes what must start at zero with an
 *                asynchronous memset on `stream`), overwritten by the call,
 *                and not to be shared by calls that overlap on the device.
 */
attn_status_t attn_fwd_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_table, int32_t block_table_stride,
                              const int32_t* seq_lens, int32_t num_seqs, int32_t max_seqlen_k,
                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                              int32_t block_size, int32_t num_blocks, float scale,
                              int32_t num_splits, attn_dtype_t dtype, attn_round_t rounding,
                              float* lse_out, void* workspace, size_t workspace_bytes,
                              int32_t* status_dev, void* stream);

/*
 * Feature-flagged variants.  "gfx942 unified attention, from the math up",
 * sec. 9, names sinks, ALiBi, softcap and sliding window among the flags a
 * dispatcher treats specially (it keeps such calls out of graph replay)
 * without defining them; this library takes their usual definitions.  With
 * diag = i + kv_len - query_len the key aligned with query row i (for decode
 * diag = kv_len - 1) and s = scale * q.k the scaled score:
 *   window_left  >= 0: key j is visible only if j >= diag - window_left;
 *                -1: unbounded.  Key tiles wholly left of every row's window
 *                are skipped, not computed and masked.
 *   window_right >= 0: key j is visible only if j <= diag + window_right;
 *                -1: unbounded (causal calls are already bounded by diag).
 *   softcap      > 0: s becomes softcap * tanh(s / softcap); 0: off.
 *   alibi_slopes NULL, or a DEVICE fp32 array [num_q_heads]: s gains
 *                -alibi_slopes[h] * |diag - j| (after the softcap).  With
 *                slopes, decode and the head-size-64/128 prefill (even
 *                query-head groups) visit the keys from the last to the first,
 *                so that the running maximum is set early; the result is the
 *                same function, summed in another order, so it is not
 *                bit-identical to a call without slopes even when they are 0.
 *   sinks        NULL, or a DEVICE fp32 array [num_q_heads]: a logit z_h that
 *                joins the softmax denominator with no value row,
 *                O = sum_j e^(s_j) V_j / (sum_j e^(s_j) + e^(z_h)); the
 *                log-sum-exp output includes it (z_h for a row with no
 *                visible key, whose output is 0).
 * Passing NULL for the whole struct, or {-1, -1, 0, NULL, NULL} with the
 * remaining fields zero, is the plain call.  Errors: window values below -1,
 * a softcap that is negative or not finite, per-head arrays that are not
 * 4-byte aligned, kv_fp8 outside {0, 1} or fp8 factors that are not finite
 * and positive give ATTN_ERR_INVALID_ARG; a missing or short fp8 prefill
 * workspace gives ATTN_ERR_WORKSPACE.  The struct is read during the call only; the
 * device arrays must stay valid until the work on `stream` has run.
 */
typedef struct {
  int32_t window_left;
  int32_t window_right;
  float softcap;
  const float* alibi_slopes;
  const float* sinks;
  /* fp8 K/V caches ([ALG] sec. 9 lists fp8 among the flags without defining
   * it; this library takes the common convention).  kv_fp8 = 1: k_cache and
   * v_cache hold OCP E4M3 codes (1 byte per element, same [num_blocks,
   * block_size, Hkv, d] layout, 16-byte aligned) and the key and value meant
   * are k_scale * code and v_scale * code; q and out keep `dtype`.  The two
   * NaN codes (S.1111.111) read as NaN: a NaN key makes the outputs of the
   * rows that see it NaN; a NaN value element makes that channel NaN in
   * every output whose tensor-core product reads it, which includes rows of
   * the same key tile that do not see the key and, in decode, the other KV
   * heads folded into the same work item (0 * NaN is NaN).  kv_fp8 = 0
   * ignores the four fields below.  k_scale and v_scale must be finite and
   * > 0.  Decode reads the codes in its kernels.  Prefill first widens the
   * pages each sequence references into `workspace` (device memory of at
   * least attn_fp8_prefill_workspace_size() bytes, 256-byte aligned, owned
   * by the caller and not touched after the work on `stream` has run), then
   * runs the 16-bit kernels on that copy.  The dense entry point takes fp8
   * K and V ([B, Sk, Hkv, d] codes whose strides, in bytes, are multiples of
   * 16) the same way, with a workspace of
   * attn_fp8_prefill_workspace_size(B, Sk, Hkv, d, Sk) bytes. */
  int32_t kv_fp8;
  float k_scale;
  float v_scale;
  void* workspace;
  size_t workspace_bytes;
} attn_features_t;

/* Bytes of `workspace` an fp8 prefill call needs: two 16-bit caches of
 * num_seqs * ceil(max_seqlen_k / block_size) pages plus their block table.
 * 0 for invalid arguments. */
size_t attn_fp8_prefill_workspace_size(int32_t num_seqs, int32_t max_seqlen_k,
                                       int32_t num_kv_heads, int32_t head_size,
                                       int32_t block_size);

/* attn_fwd_prefill, attn_fwd_dense and attn_fwd_decode with feature flags
 * (the other arguments as for those calls).  Decode keeps its kernel choice:
 * a window only narrows the key range each split reads. */
attn_status_t attn_fwd_prefill_ex(void* out, const void* q, const void* k_cache,
                                  const void* v_cache, const int32_t* block_table,
                                  int32_t block_table_stride, const int32_t* query_start_loc,
                                  const int32_t* seq_lens, int32_t num_seqs, int32_t max_seqlen_q,
                                  int32_t max_seqlen_k, int32_t total_q, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                  int32_t num_blocks, float scale, int32_t causal,
                                  attn_dtype_t dtype, attn_round_t rounding, float* lse_out,
                                  int32_t* status_dev, void* stream,
                                  const attn_features_t* features);
attn_status_t attn_fwd_dense_ex(void* out, const void* q, const void* k, const void* v,
                                const int64_t* q_strides, const int64_t* k_strides,
                                const int64_t* v_strides, const int64_t* o_strides, int32_t batch,
                                int32_t seqlen_q, int32_t seqlen_k, int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t head_size, float scale,
                                int32_t causal, attn_dtype_t dtype, attn_round_t rounding,
                                float* lse_out, int32_t* status_dev, void* stream,
                                const attn_features_t* features);
attn_status_t attn_fwd_decode_ex(void* out, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* block_table,
                                 int32_t block_table_stride, const int32_t* seq_lens,
                                 int32_t num_seqs, int32_t max_seqlen_k, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                 int32_t num_blocks, float scale, int32_t num_splits,
                                 attn_dtype_t dtype, attn_round_t rounding, float* lse_out,
                                 void* workspace, size_t workspace_bytes, int32_t* status_dev,
                                 void* stream, const attn_features_t* features);

/* Size of the device scratch array built into the library for
 * attn_fwd_decode_noalloc (16 MiB on every GPU that loads the library). */
#define ATTN_DECODE_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * attn_fwd_decode_noalloc -- attn_fwd_decode for callers that may not
 * allocate device memory.  The paper has no counterpart of this entry point;
 * it exists for this library's users.  A latency-critical serving loop cannot call
 * cudaMalloc (it may synchronise the device and has unbounded cost), and a
 * host framework whose allocator owns all device memory, or a plugin that
 * only receives input and output pointers, has no way to supply a workspace.
 * This entry point takes the same arguments as attn_fwd_decode minus the
 * workspace, runs the same kernels, and keeps the split partials in a
 * library-owned device array of ATTN_DECODE_NOALLOC_SCRATCH_BYTES.
 *
 *   - It allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - Problems whose split partials need more than the array, i.e. with
 *     attn_decode_workspace_size(num_seqs, num_q_heads, head_size, num_splits)
 *     > ATTN_DECODE_NOALLOC_SCRATCH_BYTES, are rejected with
 *     ATTN_ERR_WORKSPACE before anything is launched.
 *   - Every call looks up the array's device address in the current context
 *     (cudaGetSymbolAddress with the caller's device current; no address is
 *     kept between calls, so a device reset or another context is fine).
 *     The first call in a context may load the library's device code: make
 *     it before any stream capture.
 *   - All calls on a device share the array.  The only value that must start
 *     at zero, the work counter of the tcgen05 decode kernel, is zeroed on
 *     `stream` before each of its launches; every partial o, m and l is
 *     written before it is read.  Calls that may overlap on the device
 *     (unordered streams) race on the array and must not be issued.
 *   - It takes 16-bit caches and no feature flags (attn_fwd_decode's
 *     arguments); fp8 caches and the flags need attn_fwd_decode_ex.
 *   - Other arguments, errors and the status word: as for attn_fwd_decode.
 */
attn_status_t attn_fwd_decode_noalloc(void* out, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_table,
                                      int32_t block_table_stride, const int32_t* seq_lens,
                                      int32_t num_seqs, int32_t max_seqlen_k, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                      int32_t num_blocks, float scale, int32_t num_splits,
                                      attn_dtype_t dtype, attn_round_t rounding, float* lse_out,
                                      int32_t* status_dev, void* stream);

/*
 * attn_round_f32 -- applies the output rounding of the epilogues to n fp32
 * values: out[i] = round(in[i]) as bf16 or fp16 bit patterns (uint16_t[n]),
 * rounding in {ATTN_RTNE, ATTN_RTNA, ATTN_RTZ}.  Exposed so that the rounding
 * can be checked on its own.
 */
attn_status_t attn_round_f32(void* out, const float* in, int64_t n, attn_dtype_t dtype,
                             attn_round_t rounding, void* stream);

/* Human-readable name of a status code (static string). */
const char* attn_status_string(attn_status_t status);

/* Counters of the library's tensor-map cache (process-wide): hits are
 * encodes served from the cache, misses are encodes done by the driver.  The
 * TMA descriptors each call needs are cached on everything that defines them
 * (address, element type, sizes, strides, box, swizzle), so a repeated call on
 * the same buffers does no driver encode.  Either pointer may be NULL.
 * Diagnostic only; there is no counterpart in the pages. */
void attn_tensor_map_cache_stats(uint64_t* hits, uint64_t* misses);

/* ABI version of this header (incremented on incompatible changes; 2 added
 * the fp8 fields of attn_features_t). */
int32_t attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_FWD_H_ */

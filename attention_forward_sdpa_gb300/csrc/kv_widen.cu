// kv_widen.cu -- the first step of an fp8 prefill: the E4M3 pages that each
// sequence references are widened to the query's 16-bit format (exactly: an
// E4M3 value has 3 fraction bits and exponents 2^-9 .. 2^8, so every code is
// an fp16 normal or zero and a bf16 value) and laid out densely, page (b, p)
// at index b * pages_per_seq + p, with a matching block table.  The 16-bit
// prefill kernels then run on that copy with the K factor folded into tau
// and the V factor applied to the normalised output.  fp8 is one of the
// flags "gfx942 unified attention, from the math up" sec. 9 lists without a
// definition; the convention (per-tensor factors) is stated in attn_fwd.h.
//
// Bound: HBM.  Each referenced page is read once (1 byte per element) and
// written once (2 bytes per element); a CTA widens 4096 codes of K and of V
// of one page (grid: chunks x pages x sequences), 16-byte loads and two
// 16-byte stores per thread.

#include "attn_internal.h"
#include "e4m3.cuh"

namespace attn {
namespace {

struct WidenParams {
  const uint8_t* k8;
  const uint8_t* v8;
  const int32_t* block_table;
  const int32_t* seq_lens;
  uint16_t* k16;
  uint16_t* v16;
  int32_t* table_out;
  int32_t* status;
  int64_t page_elems;   // block_size * Hkv * d (a multiple of 64)
  int32_t bt_stride;
  int32_t pages_per_seq;
  int32_t block_size;
  int32_t num_blocks;
};

constexpr int kChunk = 256 * 16;   // codes of K (and of V) per CTA

template <bool BF16>
__global__ void __launch_bounds__(256) kv_widen_kernel(const __grid_constant__ WidenParams p) {
  const int64_t chunks = (p.page_elems + kChunk - 1) / kChunk;
  const int pg = (int)(blockIdx.x / chunks);
  const int64_t chunk = blockIdx.x % chunks;
  const int b = blockIdx.y;
  const int64_t dst_page = (int64_t)b * p.pages_per_seq + pg;
  const int sk = p.seq_lens[b];
  const int pages_b = sk > 0 ? (sk + p.block_size - 1) / p.block_size : 0;
  const bool used = pg < pages_b;
  if (chunk == 0 && threadIdx.x == 0) p.table_out[dst_page] = used ? (int32_t)dst_page : -1;
  if (!used) return;
  const int src_page = p.block_table[(int64_t)b * p.bt_stride + pg];
  const bool ok = src_page >= 0 && src_page < p.num_blocks;
  if (!ok && chunk == 0 && threadIdx.x == 0) report_status(p.status, kStatusBadBlockTable);
  const int64_t i = (chunk * kChunk) / 16 + threadIdx.x;   // 16-code group within the page
  if (i * 16 >= p.page_elems) return;
  const int64_t src = (int64_t)(ok ? src_page : 0) * p.page_elems / 16 + i;
  uint4 klo = make_uint4(0u, 0u, 0u, 0u), khi = klo, vlo = klo, vhi = klo;
  if (ok) {
    e4m3x16_widen<BF16>(__ldg(reinterpret_cast<const uint4*>(p.k8) + src), klo, khi);
    e4m3x16_widen<BF16>(__ldg(reinterpret_cast<const uint4*>(p.v8) + src), vlo, vhi);
  }
  uint4* kd = reinterpret_cast<uint4*>(p.k16) + (dst_page * p.page_elems / 16 + i) * 2;
  uint4* vd = reinterpret_cast<uint4*>(p.v16) + (dst_page * p.page_elems / 16 + i) * 2;
  kd[0] = klo;
  kd[1] = khi;
  vd[0] = vlo;
  vd[1] = vhi;
}

// Dense fp8 input: K and V as logical [B, Sk, Hkv, d] E4M3 codes with any
// (batch, row, head) strides (bytes, multiples of 16; channels contiguous)
// widened into contiguous 16-bit [B, Sk, Hkv, d] copies.  One thread per 16
// codes of K and of V.
struct WidenDenseParams {
  const uint8_t* k8;
  const uint8_t* v8;
  uint16_t* k16;
  uint16_t* v16;
  int64_t ks[3], vs[3];   // source strides (elements = bytes): batch, row, head
  int64_t groups;         // B * Sk * Hkv * d / 16
  int32_t seqlen_k, num_kv_heads, head_size;
};

template <bool BF16>
__global__ void __launch_bounds__(256) kv_widen_dense_kernel(const __grid_constant__ WidenDenseParams p) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= p.groups) return;
  const int per_row = p.head_size / 16;
  const int64_t row = i / per_row;                 // ((b * Sk) + s) * Hkv + h
  const int c16 = (int)(i % per_row);
  const int h = (int)(row % p.num_kv_heads);
  const int64_t bs = row / p.num_kv_heads;
  const int s = (int)(bs % p.seqlen_k);
  const int64_t b = bs / p.seqlen_k;
  const int64_t ko = b * p.ks[0] + s * p.ks[1] + h * p.ks[2] + 16 * c16;
  const int64_t vo = b * p.vs[0] + s * p.vs[1] + h * p.vs[2] + 16 * c16;
  uint4 klo, khi, vlo, vhi;
  e4m3x16_widen<BF16>(__ldg(reinterpret_cast<const uint4*>(p.k8 + ko)), klo, khi);
  e4m3x16_widen<BF16>(__ldg(reinterpret_cast<const uint4*>(p.v8 + vo)), vlo, vhi);
  uint4* kd = reinterpret_cast<uint4*>(p.k16) + 2 * i;
  uint4* vd = reinterpret_cast<uint4*>(p.v16) + 2 * i;
  kd[0] = klo;
  kd[1] = khi;
  vd[0] = vlo;
  vd[1] = vhi;
}

}  // namespace

cudaError_t launch_kv_widen_dense(const void* k8, const void* v8, const int64_t* k_strides,
                                  const int64_t* v_strides, int32_t batch, int32_t seqlen_k,
                                  int32_t num_kv_heads, int32_t head_size, bool bf16, void* k16,
                                  void* v16, cudaStream_t stream) {
  WidenDenseParams p;
  p.k8 = static_cast<const uint8_t*>(k8);
  p.v8 = static_cast<const uint8_t*>(v8);
  p.k16 = static_cast<uint16_t*>(k16);
  p.v16 = static_cast<uint16_t*>(v16);
  for (int i = 0; i < 3; ++i) {
    p.ks[i] = k_strides[i];
    p.vs[i] = v_strides[i];
  }
  p.seqlen_k = seqlen_k;
  p.num_kv_heads = num_kv_heads;
  p.head_size = head_size;
  p.groups = (int64_t)batch * seqlen_k * num_kv_heads * (head_size / 16);
  if (p.groups == 0) return cudaSuccess;
  const int64_t blocks = (p.groups + 255) / 256;
  if (blocks > 2147483647) return cudaErrorInvalidValue;
  if (bf16) kv_widen_dense_kernel<true><<<(unsigned)blocks, 256, 0, stream>>>(p);
  else kv_widen_dense_kernel<false><<<(unsigned)blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_kv_widen(const void* k8, const void* v8, const int32_t* block_table,
                            int32_t bt_stride, const int32_t* seq_lens, int32_t num_seqs,
                            int32_t pages_per_seq, int32_t block_size, int32_t num_blocks,
                            int64_t page_elems, bool bf16, void* k16, void* v16,
                            int32_t* table_out, int32_t* status, cudaStream_t stream) {
  WidenParams p;
  p.k8 = static_cast<const uint8_t*>(k8);
  p.v8 = static_cast<const uint8_t*>(v8);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.k16 = static_cast<uint16_t*>(k16);
  p.v16 = static_cast<uint16_t*>(v16);
  p.table_out = table_out;
  p.status = status;
  p.page_elems = page_elems;
  p.bt_stride = bt_stride;
  p.pages_per_seq = pages_per_seq;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  const int64_t chunks = (page_elems + kChunk - 1) / kChunk;
  if ((int64_t)pages_per_seq * chunks > 2147483647) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)(pages_per_seq * chunks), (unsigned)num_seqs);
  if (bf16) kv_widen_kernel<true><<<grid, 256, 0, stream>>>(p);
  else kv_widen_kernel<false><<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace attn

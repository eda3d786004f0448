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
// written once (2 bytes per element); one CTA per (page, sequence), 16-byte
// loads and 2 x 16-byte stores per thread step.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn_internal.h"

namespace attn {
namespace {

// Two E4M3 codes (low byte -> low half) to f16x2: the hardware conversion is
// exact for this direction.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t h;
  const uint16_t c = (uint16_t)two_codes;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(c));
  return h;
}

// f16x2 holding E4M3 values -> bf16x2 (exact: at most 4 significant bits).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
  return *reinterpret_cast<const uint32_t*>(&b);
}

template <bool BF16>
__device__ __forceinline__ uint32_t widen_pair(uint32_t two_codes) {
  const uint32_t h = e4m3x2_to_f16x2(two_codes);
  return BF16 ? f16x2_to_bf16x2(h) : h;
}

// 16 codes -> 16 16-bit values (element order kept)
template <bool BF16>
__device__ __forceinline__ void widen16(const uint4 w, uint4& lo, uint4& hi) {
  lo.x = widen_pair<BF16>(w.x);
  lo.y = widen_pair<BF16>(w.x >> 16);
  lo.z = widen_pair<BF16>(w.y);
  lo.w = widen_pair<BF16>(w.y >> 16);
  hi.x = widen_pair<BF16>(w.z);
  hi.y = widen_pair<BF16>(w.z >> 16);
  hi.z = widen_pair<BF16>(w.w);
  hi.w = widen_pair<BF16>(w.w >> 16);
}

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

template <bool BF16>
__global__ void __launch_bounds__(256) kv_widen_kernel(const __grid_constant__ WidenParams p) {
  const int pg = blockIdx.x;
  const int b = blockIdx.y;
  const int64_t dst_page = (int64_t)b * p.pages_per_seq + pg;
  const int sk = p.seq_lens[b];
  const int pages_b = sk > 0 ? (sk + p.block_size - 1) / p.block_size : 0;
  const bool used = pg < pages_b && pg < p.pages_per_seq;
  if (threadIdx.x == 0) p.table_out[dst_page] = used ? (int32_t)dst_page : -1;
  if (!used) return;
  const int src_page = p.block_table[(int64_t)b * p.bt_stride + pg];
  const bool ok = src_page >= 0 && src_page < p.num_blocks;
  if (!ok && threadIdx.x == 0) report_status(p.status, kStatusBadBlockTable);
  const uint4* ks = reinterpret_cast<const uint4*>(p.k8 + (int64_t)(ok ? src_page : 0) * p.page_elems);
  const uint4* vs = reinterpret_cast<const uint4*>(p.v8 + (int64_t)(ok ? src_page : 0) * p.page_elems);
  uint4* kd = reinterpret_cast<uint4*>(p.k16 + dst_page * p.page_elems);
  uint4* vd = reinterpret_cast<uint4*>(p.v16 + dst_page * p.page_elems);
  const int64_t n16 = p.page_elems / 16;
  for (int64_t i = threadIdx.x; i < n16; i += blockDim.x) {
    uint4 klo = make_uint4(0u, 0u, 0u, 0u), khi = klo, vlo = klo, vhi = klo;
    if (ok) {
      widen16<BF16>(__ldg(ks + i), klo, khi);
      widen16<BF16>(__ldg(vs + i), vlo, vhi);
    }
    kd[2 * i] = klo;
    kd[2 * i + 1] = khi;
    vd[2 * i] = vlo;
    vd[2 * i + 1] = vhi;
  }
}

}  // namespace

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
  const dim3 grid((unsigned)pages_per_seq, (unsigned)num_seqs);
  if (bf16) kv_widen_kernel<true><<<grid, 256, 0, stream>>>(p);
  else kv_widen_kernel<false><<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace attn

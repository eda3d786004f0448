"""Seeded synthetic inputs for the paged SDPA forward.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path's tests/benchmark and the oracle read
the same 16-bit tensors it produces.

Layout (the paged-KV layout of "gfx942 unified attention, from the math up",
sec. 5):
  q            [total_q, Hq, d]              packed queries, 16-bit
  k_cache      [num_blocks, block_size, Hkv, d]
  v_cache      [num_blocks, block_size, Hkv, d]
  block_table  [num_seqs, max_pages] int32   page ids; unused entries are -1
  query_start_loc [num_seqs + 1] int32       prefix sum of query lengths
  seq_lens     [num_seqs] int32              kv length per sequence

Recipe (fixed draw order, three independent generators derived from the seed):
  1. lengths    -- torch.Generator(seed): kv lengths uniform in [lo, hi] when a
                   range is asked for;
  2. layout     -- torch.Generator(seed + 1000003): a random permutation of the
                   page pool (when ``permute``);
  3. values     -- torch.Generator(seed + 2000006): Q, then per sequence the
                   logical K [Sk, Hkv, d], then the logical V, each randn * sigma
                   in fp32, rounded to the 16-bit dtype by round-to-nearest-even.
Because the values are drawn in logical order, the same seed gives the same
logical K/V whatever the block size and permutation.  Pages that no table
references are filled with NaN, and so are the slots past kv_len in a
sequence's last page, so that any read outside the visible keys shows up.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

LAYOUT_SALT = 1000003
VALUE_SALT = 2000006


@dataclass
class PagedProblem:
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_table: torch.Tensor
    query_start_loc: torch.Tensor
    seq_lens: torch.Tensor
    q_lens: list
    kv_lens: list
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    dtype: torch.dtype
    scale: float
    causal: bool
    meta: dict = field(default_factory=dict)
    # fp8 caches: K and V hold float8_e4m3fn codes and the values meant are
    # code * k_scale and code * v_scale (1.0 for 16-bit caches)
    k_scale: float = 1.0
    v_scale: float = 1.0

    @property
    def kv_fp8(self) -> bool:
        return self.k_cache.dtype == torch.float8_e4m3fn

    @property
    def num_seqs(self) -> int:
        return len(self.kv_lens)

    @property
    def total_q(self) -> int:
        return int(sum(self.q_lens))

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_seqlen_q(self) -> int:
        return int(max(self.q_lens)) if self.q_lens else 0

    @property
    def max_seqlen_k(self) -> int:
        return int(max(self.kv_lens)) if self.kv_lens else 0


def _poison_value(dtype: torch.dtype) -> float:
    return float("nan")


def paged_problem(*, seed: int, q_lens, kv_lens, num_q_heads: int, num_kv_heads: int,
                  head_size: int, block_size: int, dtype: torch.dtype = torch.bfloat16,
                  sigma: float = 1.0, causal: bool = True, scale: float | None = None,
                  permute: bool = True, pool_extra: int = 0, poison: bool = True,
                  table_pad: int = 0, kv_dtype: torch.dtype | None = None) -> PagedProblem:
    """Builds one paged problem on the CPU.  ``q_lens``/``kv_lens`` are lists of
    per-sequence lengths.  ``pool_extra`` unreferenced pages are added to the
    pool; ``table_pad`` extra -1 columns are added to the block table.
    ``kv_dtype=torch.float8_e4m3fn`` stores the caches as fp8 codes: the same
    fp32 draws divided by a per-tensor factor sigma * 6 / 448 (so +-6 sigma
    spans the format), clamped to +-448 and rounded to nearest-even; the
    factor is returned as ``k_scale`` / ``v_scale``."""
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    assert len(q_lens) == len(kv_lens)
    bs = int(block_size)
    pages = [max(0, -(-k // bs)) for k in kv_lens]
    n_pages = sum(pages) + int(pool_extra)
    max_pages = max(pages) if pages else 0
    max_pages = max(1, max_pages + int(table_pad))

    g_layout = torch.Generator().manual_seed(seed + LAYOUT_SALT)
    g_val = torch.Generator().manual_seed(seed + VALUE_SALT)

    if permute and n_pages > 0:
        perm = torch.randperm(n_pages, generator=g_layout)
    else:
        perm = torch.arange(n_pages)
    block_table = torch.full((len(kv_lens), max_pages), -1, dtype=torch.int32)
    cursor = 0
    for b, npg in enumerate(pages):
        block_table[b, :npg] = perm[cursor:cursor + npg].to(torch.int32)
        cursor += npg

    H, Hk, d = num_q_heads, num_kv_heads, head_size
    total_q = sum(q_lens)
    q = (torch.randn((total_q, H, d), generator=g_val, dtype=torch.float32) * sigma).to(dtype)

    fp8 = kv_dtype == torch.float8_e4m3fn
    if kv_dtype is not None and not fp8 and kv_dtype != dtype:
        raise ValueError("kv_dtype is the query dtype or float8_e4m3fn")
    cdt = torch.float8_e4m3fn if fp8 else dtype
    kv_scale = sigma * 6.0 / 448.0 if fp8 else 1.0
    fill = _poison_value(dtype) if poison else 0.0
    k_cache = torch.full((max(n_pages, 1), bs, Hk, d), fill, dtype=cdt)
    v_cache = torch.full((max(n_pages, 1), bs, Hk, d), fill, dtype=cdt)
    for name, cache in (("k", k_cache), ("v", v_cache)):
        for b, sk in enumerate(kv_lens):
            if sk == 0:
                continue
            vals = torch.randn((sk, Hk, d), generator=g_val, dtype=torch.float32) * sigma
            if fp8:
                vals = (vals / kv_scale).clamp(-448.0, 448.0).to(cdt)
            else:
                vals = vals.to(dtype)
            npg = pages[b]
            ids = block_table[b, :npg].long()
            padded = torch.full((npg * bs, Hk, d), fill, dtype=cdt)
            padded[:sk] = vals
            cache[ids] = padded.view(npg, bs, Hk, d)

    qsl = torch.zeros(len(q_lens) + 1, dtype=torch.int32)
    if q_lens:
        qsl[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int64), 0).to(torch.int32)
    seq_lens = torch.tensor(kv_lens, dtype=torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(head_size)
    return PagedProblem(q=q, k_cache=k_cache, v_cache=v_cache, block_table=block_table,
                        query_start_loc=qsl, seq_lens=seq_lens, q_lens=q_lens,
                        kv_lens=kv_lens, num_q_heads=H, num_kv_heads=Hk, head_size=d,
                        block_size=bs, dtype=dtype, scale=float(scale), causal=bool(causal),
                        meta={"seed": seed, "sigma": sigma, "permute": permute},
                        k_scale=float(kv_scale), v_scale=float(kv_scale))


def random_kv_lens(seed: int, n: int, lo: int, hi: int) -> list:
    """n kv lengths uniform on [lo, hi] from torch.Generator(seed) (draw 1)."""
    g = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


# --------------------------------------------------------------------------
# The named workloads.  Shapes follow the five measured configurations:
# --------------------------------------------------------------------------

def workload(name: str, seed: int = 0, **over) -> PagedProblem:
    """Named workloads (sizes as stated):
      prefill_causal_fp16_s128_d64   causal, fp16, B=1, Hq=Hkv=2, Sq=Sk=128, d=64,
                                     one page of 128, tau = 1/8, N(0,1)
      prefill_causal_bf16_gqa_s2048  causal, bf16, B=1, Hq=32, Hkv=8, Sq=Sk=2048,
                                     d=128, block_size 64, permuted table, N(0,1)
      decode_bf16_b64_paged16        decode (Sq=1), bf16, B=64, Hq=32, Hkv=8,
                                     d=128, Sk ~ U[512, 8192], block_size 16,
                                     shared permuted pool, N(0,1)
      prefill_causal_bf16_s8192      causal, bf16, B=1, Sq=Sk=8192, Hq=32, Hkv=8,
                                     d=128, block_size 64, N(0, 0.5^2)
      prefill_chunked_bf16_b4        chunked causal, bf16, B=4, Sq=512, Sk=8192,
                                     Hq=32, Hkv=8, d=128, block_size 64, N(0, 0.5^2)
      dense_bf16_bshd_s16384         non-causal, bf16, BSHD, B=4, H=16, S=16384,
                                     d=128, one page per sequence, N(0,1)
      prefill_causal_bf16_gqa_s2048_d256   the 2048 workload at head size 256
      prefill_causal_bf16_s8192_d256       the 8192 workload at head size 256
      decode_bf16_b64_paged16_d64 / _d256  the decode workload at head size 64 / 256
    Keyword overrides replace any argument of paged_problem (e.g. smaller
    lengths for parity runs at reduced size)."""
    if name == "prefill_causal_fp16_s128_d64":
        kw = dict(q_lens=[128], kv_lens=[128], num_q_heads=2, num_kv_heads=2, head_size=64,
                  block_size=128, dtype=torch.float16, sigma=1.0, causal=True, scale=1.0 / 8,
                  permute=False)
    elif name == "prefill_causal_bf16_gqa_s2048":
        kw = dict(q_lens=[2048], kv_lens=[2048], num_q_heads=32, num_kv_heads=8, head_size=128,
                  block_size=64, dtype=torch.bfloat16, sigma=1.0, causal=True)
    elif name == "decode_bf16_b64_paged16":
        lens = random_kv_lens(seed, 64, 512, 8192)
        kw = dict(q_lens=[1] * 64, kv_lens=lens, num_q_heads=32, num_kv_heads=8, head_size=128,
                  block_size=16, dtype=torch.bfloat16, sigma=1.0, causal=False)
    elif name == "prefill_causal_bf16_s8192":
        kw = dict(q_lens=[8192], kv_lens=[8192], num_q_heads=32, num_kv_heads=8, head_size=128,
                  block_size=64, dtype=torch.bfloat16, sigma=0.5, causal=True)
    elif name == "prefill_chunked_bf16_b4":
        kw = dict(q_lens=[512] * 4, kv_lens=[8192] * 4, num_q_heads=32, num_kv_heads=8,
                  head_size=128, block_size=64, dtype=torch.bfloat16, sigma=0.5, causal=True)
    elif name == "dense_bf16_bshd_s16384":
        kw = dict(q_lens=[16384] * 4, kv_lens=[16384] * 4, num_q_heads=16, num_kv_heads=16,
                  head_size=128, block_size=16384, dtype=torch.bfloat16, sigma=1.0, causal=False,
                  permute=False, poison=False)
    elif name in ("prefill_causal_bf16_gqa_s2048_d256", "prefill_causal_bf16_s8192_d256",
                  "decode_bf16_b64_paged16_d256"):
        return workload(name[:-len("_d256")], seed=seed, **{"head_size": 256, **over})
    elif name == "decode_bf16_b64_paged16_d64":
        return workload("decode_bf16_b64_paged16", seed=seed, **{"head_size": 64, **over})
    else:
        raise KeyError(name)
    kw.update(over)
    return paged_problem(seed=seed, **kw)


WORKLOADS = ("prefill_causal_fp16_s128_d64", "prefill_causal_bf16_gqa_s2048",
             "decode_bf16_b64_paged16", "prefill_causal_bf16_s8192",
             "prefill_chunked_bf16_b4", "dense_bf16_bshd_s16384",
             "prefill_causal_bf16_gqa_s2048_d256", "prefill_causal_bf16_s8192_d256",
             "decode_bf16_b64_paged16_d64", "decode_bf16_b64_paged16_d256")

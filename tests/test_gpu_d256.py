"""GPU parity at head size 256 (prefill_d256_tcgen05.cu for prefill and the
dense entry point, the SIMT split kernel for decode) against the fp64 oracle.

Tolerance: 2e-2 (fp16) / 4e-2 (bf16) max |err| per element, as for the other
head sizes ("gfx942 unified attention, from the math up", sec. 10).  The cases
span every block size (one to eight pages per key tile, and pages longer than
a tile), ragged query and key tails, GQA with odd and even groups, causal and
non-causal, rows that see no key, several key tiles (so that the five-slot
K/V ring wraps), score scales large enough to move the running max after the
first tile (the O rescale that waits for the previous P.V product), the three
output roundings against the oracle's rounding of the kernel's own fp32
result, the log-sum-exp, bit identity across runs, paging invariance, and the
dense BSHD / BHSD entry point against the paged one.
"""
import numpy as np
import pytest
import torch

import attn_inputs
from oracle import oracle
from tests.helpers import (TOL, as_rows, gpu_decode, gpu_prefill, max_err, oracle_run, sample_rows,
                           to_dev, worst)
from tests.test_gpu_dense import make, run_dense

pytestmark = pytest.mark.gpu


def check(prob, out):
    torch.cuda.synchronize()
    ref, _ = oracle_run(prob)
    got = as_rows(out)
    err = max_err(got, ref)
    assert err <= TOL[prob.dtype], (err, worst(got, ref))


CASES = {
    "gqa4_bf16_bs64_varlen_causal": dict(q_lens=[300, 1, 129, 77], kv_lens=[300, 500, 129, 1000],
                                         num_q_heads=8, num_kv_heads=2, block_size=64,
                                         dtype=torch.bfloat16, causal=True),
    "gqa4_bf16_bs64_varlen_noncausal": dict(q_lens=[300, 1, 129, 77], kv_lens=[300, 500, 129, 1000],
                                            num_q_heads=8, num_kv_heads=2, block_size=64,
                                            dtype=torch.bfloat16, causal=False),
    "mha_fp16_bs128_noncausal": dict(q_lens=[200, 5], kv_lens=[333, 1000], num_q_heads=2,
                                     num_kv_heads=2, block_size=128, dtype=torch.float16,
                                     causal=False),
    "gqa3_bf16_bs16_causal": dict(q_lens=[130, 40], kv_lens=[400, 40], num_q_heads=6,
                                  num_kv_heads=2, block_size=16, dtype=torch.bfloat16, causal=True),
    "gqa2_fp16_bs32_causal": dict(q_lens=[70, 300], kv_lens=[90, 300], num_q_heads=4,
                                  num_kv_heads=2, block_size=32, dtype=torch.float16, causal=True),
    "gqa8_bf16_bs256_noncausal_sigma2": dict(q_lens=[250, 3], kv_lens=[700, 513], num_q_heads=16,
                                             num_kv_heads=2, block_size=256, dtype=torch.bfloat16,
                                             causal=False, sigma=2.0),
    "mha_bf16_bs128_long_causal_sigma2": dict(q_lens=[1000], kv_lens=[1000], num_q_heads=3,
                                              num_kv_heads=3, block_size=128, dtype=torch.bfloat16,
                                              causal=True, sigma=2.0),
    "gqa2_fp16_bs64_chunked": dict(q_lens=[100, 256], kv_lens=[900, 700], num_q_heads=4,
                                   num_kv_heads=2, block_size=64, dtype=torch.float16, causal=True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_d256_matches_oracle(name):
    prob = attn_inputs.paged_problem(seed=61, head_size=256, pool_extra=5, **CASES[name])
    check(prob, gpu_prefill(prob))


def test_rows_without_keys_and_lse():
    prob = attn_inputs.paged_problem(seed=62, q_lens=[200, 5, 3], kv_lens=[50, 0, 140],
                                     num_q_heads=4, num_kv_heads=2, head_size=256, block_size=32,
                                     causal=True)
    out, lse = gpu_prefill(prob, lse=True)
    torch.cuda.synchronize()
    ref, ref_lse = oracle_run(prob)
    got = as_rows(out)
    assert max_err(got, ref) <= TOL[prob.dtype]
    g = lse.cpu().numpy().reshape(-1).astype(np.float64)
    empty = np.isinf(ref_lse)
    assert empty.sum() > 0
    assert np.all(np.isneginf(g[empty])) and np.all(got[empty] == 0)
    assert np.max(np.abs(g[~empty] - ref_lse[~empty])) < 2e-3


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_rounding_modes(dtype):
    """RTNE / RTNA / RTZ must equal the oracle's rounding of the kernel's own
    fp32 result (the result is deterministic)."""
    prob = attn_inputs.paged_problem(seed=63, q_lens=[300, 45], kv_lens=[300, 600], num_q_heads=4,
                                     num_kv_heads=2, head_size=256, block_size=64, dtype=dtype,
                                     causal=False, sigma=3.0)
    t = to_dev(prob)
    x = gpu_prefill(prob, t, rounding=3)
    torch.cuda.synchronize()
    xf = x.cpu().numpy().astype(np.float32)
    ref, _ = oracle_run(prob)
    assert max_err(xf.reshape(-1, 256).astype(np.float64), ref) <= TOL[dtype]
    odt = oracle.BF16 if dtype == torch.bfloat16 else oracle.F16
    for mode in (0, 1, 2):
        r = gpu_prefill(prob, t, rounding=mode)
        torch.cuda.synchronize()
        got = r.cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, oracle.round_f32(xf, odt, mode)), mode


def test_bit_identical_runs_and_paging():
    outs = []
    for bs, perm in ((64, True), (16, True), (128, False), (256, True), (64, True)):
        prob = attn_inputs.paged_problem(seed=64, q_lens=[300, 77], kv_lens=[520, 77], num_q_heads=4,
                                         num_kv_heads=2, head_size=256, block_size=bs, causal=True,
                                         permute=perm, pool_extra=3)
        outs.append(gpu_prefill(prob))
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(outs[0], o)


# Odd and even groups, one to four pages per key tile: every query head reads
# its KV head's pages, so the GQA result equals the MHA one on materialised K/V
# bit for bit.
@pytest.mark.parametrize("hq,bs", [(6, 64), (8, 64), (8, 16), (4, 256)])
def test_gqa_equals_materialised_mha(hq, bs):
    g = attn_inputs.paged_problem(seed=65, q_lens=[260, 900], kv_lens=[300, 1000], num_q_heads=hq,
                                  num_kv_heads=2, head_size=256, block_size=bs, causal=True)
    m = attn_inputs.paged_problem(seed=65, q_lens=[260, 900], kv_lens=[300, 1000], num_q_heads=hq,
                                  num_kv_heads=hq, head_size=256, block_size=bs, causal=True)
    m.q = g.q.clone()
    m.k_cache = g.k_cache.repeat_interleave(hq // 2, dim=2).contiguous()
    m.v_cache = g.v_cache.repeat_interleave(hq // 2, dim=2).contiguous()
    m.block_table = g.block_table.clone()
    a, b = gpu_prefill(g), gpu_prefill(m)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_bad_block_table_entry_is_reported():
    prob = attn_inputs.paged_problem(seed=66, q_lens=[130], kv_lens=[300], num_q_heads=2,
                                     num_kv_heads=1, head_size=256, block_size=64, causal=True)
    prob.block_table[0, 2] = prob.num_blocks + 1000
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_prefill(prob, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5


def test_long_causal_sampled():
    """Sq = Sk = 4096, GQA 4:1, 16 key tiles per heaviest row block."""
    prob = attn_inputs.paged_problem(seed=67, q_lens=[4096], kv_lens=[4096], num_q_heads=8,
                                     num_kv_heads=2, head_size=256, block_size=64, causal=True,
                                     sigma=0.5)
    out = gpu_prefill(prob)
    torch.cuda.synchronize()
    rows = sample_rows(prob, per_head_random=24)
    ref, _ = oracle_run(prob, rows=rows)
    got = as_rows(out)[rows]
    assert max_err(got, ref) <= TOL[prob.dtype], worst(got, ref)


# ---------------------------------------------------------------- dense entry

@pytest.mark.parametrize("layout", ["bshd", "bhsd"])
@pytest.mark.parametrize("causal", [True, False])
def test_dense_d256_matches_oracle_and_paged(layout, causal):
    B, Sq, Sk, Hq, Hkv = 2, 200, 384, 4, 2
    prob = make(B, Sq, Sk, Hq, Hkv, 256, torch.bfloat16, causal, seed=68)
    out, lse = run_dense(prob, B, Sq, Sk, layout, lse=True)
    ref_out, ref_lse = gpu_prefill(prob, lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    assert torch.equal(lse, ref_lse.view(B, Sq, Hq).transpose(1, 2))
    ref, _ = oracle_run(prob)
    assert max_err(as_rows(out), ref) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("layout", ["bshd", "bhsd"])
def test_dense_d256_ragged_keys_padded_strides(layout):
    B, Sq, Sk = 3, 129, 77
    prob = make(B, Sq, Sk, 2, 1, 256, torch.float16, False, seed=69)
    out = run_dense(prob, B, Sq, Sk, layout, pad=8)
    torch.cuda.synchronize()
    ref, _ = oracle_run(prob)
    assert max_err(as_rows(out), ref) <= TOL[torch.float16]


# ---------------------------------------------------------------- decode

@pytest.mark.parametrize("splits", [1, 3, 8])
@pytest.mark.parametrize("hq,hkv", [(8, 2), (6, 2), (16, 2), (4, 4)])
def test_decode_d256(splits, hq, hkv):
    prob = attn_inputs.paged_problem(seed=70, q_lens=[1] * 5, kv_lens=[1, 16, 0, 300, 2049],
                                     num_q_heads=hq, num_kv_heads=hkv, head_size=256,
                                     block_size=16, causal=False, pool_extra=4)
    check(prob, gpu_decode(prob, splits=splits))


def test_decode_d256_fp16_rounding_and_lse():
    prob = attn_inputs.paged_problem(seed=71, q_lens=[1] * 3, kv_lens=[130, 9, 2500],
                                     num_q_heads=8, num_kv_heads=2, head_size=256, block_size=32,
                                     dtype=torch.float16, causal=False, sigma=2.0)
    t = to_dev(prob)
    x = gpu_decode(prob, t, splits=8, rounding=3)
    out, lse = gpu_decode(prob, t, splits=8, rounding=2, lse=True)
    torch.cuda.synchronize()
    ref, ref_lse = oracle_run(prob)
    assert max_err(x.cpu().numpy().reshape(-1, 256).astype(np.float64), ref) <= TOL[torch.float16]
    xf = x.cpu().numpy().astype(np.float32)
    got = out.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, oracle.round_f32(xf, oracle.F16, 2))
    assert np.max(np.abs(lse.cpu().numpy().reshape(-1) - ref_lse)) < 2e-3

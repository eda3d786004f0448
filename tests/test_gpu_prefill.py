"""GPU parity of the tcgen05 prefill / dense forward against the fp64 oracle.

Tolerance (max |err| per element vs the fp64 oracle): 2e-2 for fp16 and 4e-2
for bf16, the correctness gate of "gfx942 unified attention, from the math
up", sec. 10.  Small cases compare every element; the full-size workloads
compare the full tensor for the 128, 2048 and chunked workloads and a row
sample for the 8192 and dense ones (every sequence and head: first, second,
last two rows and 256 random rows -- rows are independent, so each sampled
row is exact).
Also: a batch of 300 short sequences, run-to-run bit identity, invariance to
paging (block size and permutation), GQA vs materialised MHA, rows without
visible keys, and the epilogue rounding against the oracle's rounding of the
kernel's own fp32 result.
"""
import numpy as np
import pytest
import torch

import attn_inputs
from tests.helpers import (TOL, as_rows, gpu_prefill, max_err, oracle_run, record, sample_rows,
                           to_dev, worst)
from oracle import oracle

pytestmark = pytest.mark.gpu


def check_full(prob, name=None, **kw):
    out = gpu_prefill(prob, **kw)
    torch.cuda.synchronize()
    ref, _ = oracle_run(prob)
    got = as_rows(out)
    if name:
        record(name, got, ref, prob.dtype)
    err = max_err(got, ref)
    assert err <= TOL[prob.dtype], (err, worst(got, ref))
    return out


SMALL = {
    "gqa4_bf16_d128_bs64_varlen_causal": dict(q_lens=[300, 1, 129, 77], kv_lens=[300, 500, 129, 1000],
                                              num_q_heads=8, num_kv_heads=2, head_size=128,
                                              block_size=64, dtype=torch.bfloat16, causal=True),
    "gqa4_bf16_d128_bs64_varlen_noncausal": dict(q_lens=[300, 1, 129, 77], kv_lens=[300, 500, 129, 1000],
                                                 num_q_heads=8, num_kv_heads=2, head_size=128,
                                                 block_size=64, dtype=torch.bfloat16, causal=False),
    "mha_fp16_d64_bs128_causal": dict(q_lens=[128, 257], kv_lens=[128, 300], num_q_heads=2,
                                      num_kv_heads=2, head_size=64, block_size=128,
                                      dtype=torch.float16, causal=True, scale=0.125),
    "gqa3_bf16_d128_bs32_causal": dict(q_lens=[130, 40], kv_lens=[400, 40], num_q_heads=6,
                                       num_kv_heads=2, head_size=128, block_size=32,
                                       dtype=torch.bfloat16, causal=True),
    "gqa2_fp16_d128_bs16_causal": dict(q_lens=[70, 300], kv_lens=[90, 300], num_q_heads=4,
                                       num_kv_heads=2, head_size=128, block_size=16,
                                       dtype=torch.float16, causal=True),
    "gqa8_bf16_d64_bs256_noncausal": dict(q_lens=[250, 3], kv_lens=[700, 513], num_q_heads=16,
                                          num_kv_heads=2, head_size=64, block_size=256,
                                          dtype=torch.bfloat16, causal=False),
    "mha_bf16_d128_bs128_long_causal": dict(q_lens=[1000], kv_lens=[1000], num_q_heads=3,
                                            num_kv_heads=3, head_size=128, block_size=128,
                                            dtype=torch.bfloat16, causal=True, sigma=2.0),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_cases_match_oracle(name):
    prob = attn_inputs.paged_problem(seed=21, pool_extra=5, **SMALL[name])
    check_full(prob)


@pytest.mark.parametrize("d,causal,bs", [(128, True, 64), (128, False, 16), (64, True, 128),
                                         (256, True, 32)])
def test_many_sequences(d, causal, bs):
    """A batch of 300 short sequences (some with no query rows, some with no
    keys): one grid row per sequence, most CTAs of the longest row block exit
    at once."""
    rng = np.random.default_rng(d + bs)
    q_lens = [int(x) for x in rng.integers(0, 140, size=300)]
    q_lens[7] = 0
    kv_lens = [q + int(rng.integers(0, 40)) for q in q_lens]
    kv_lens[11] = 0
    q_lens[11] = 0 if causal else q_lens[11]
    prob = attn_inputs.paged_problem(seed=40 + d, q_lens=q_lens, kv_lens=kv_lens, num_q_heads=4,
                                     num_kv_heads=2, head_size=d, block_size=bs, causal=causal,
                                     pool_extra=3)
    check_full(prob)


def test_query_longer_than_keys_gives_zero_rows():
    prob = attn_inputs.paged_problem(seed=22, q_lens=[200, 5], kv_lens=[50, 0], num_q_heads=4,
                                     num_kv_heads=2, head_size=128, block_size=64, causal=True)
    out, lse = gpu_prefill(prob, lse=True)
    torch.cuda.synchronize()
    ref, ref_lse = oracle_run(prob)
    got = as_rows(out)
    assert max_err(got, ref) <= TOL[prob.dtype]
    lse_h = lse.cpu().numpy().reshape(-1).astype(np.float64)
    empty = np.isinf(ref_lse)
    assert empty.sum() > 0
    assert np.all(np.isneginf(lse_h[empty]))
    assert np.all(got[empty] == 0)
    assert np.max(np.abs(lse_h[~empty] - ref_lse[~empty])) < 2e-3


def test_noncausal_zero_keys():
    prob = attn_inputs.paged_problem(seed=23, q_lens=[5, 130], kv_lens=[0, 7], num_q_heads=2,
                                     num_kv_heads=1, head_size=64, block_size=16, causal=False)
    check_full(prob)


def test_lse_matches_oracle():
    prob = attn_inputs.paged_problem(seed=24, q_lens=[256, 100], kv_lens=[256, 700], num_q_heads=8,
                                     num_kv_heads=2, head_size=128, block_size=64, causal=True)
    out, lse = gpu_prefill(prob, lse=True)
    torch.cuda.synchronize()
    _, ref_lse = oracle_run(prob)
    assert np.max(np.abs(lse.cpu().numpy().reshape(-1) - ref_lse)) < 2e-3


def test_run_to_run_bit_identical():
    prob = attn_inputs.paged_problem(seed=25, q_lens=[700, 300], kv_lens=[900, 300], num_q_heads=8,
                                     num_kv_heads=2, head_size=128, block_size=64, causal=True)
    t = to_dev(prob)
    a = gpu_prefill(prob, t)
    b = gpu_prefill(prob, t)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_paging_invariance_bit_identical():
    outs = []
    for bs, perm in ((64, True), (16, True), (128, False), (256, True)):
        prob = attn_inputs.paged_problem(seed=26, q_lens=[300, 77], kv_lens=[520, 77], num_q_heads=4,
                                         num_kv_heads=2, head_size=128, block_size=bs, causal=True,
                                         permute=perm, pool_extra=3)
        outs.append(gpu_prefill(prob))
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(outs[0], o)


def test_gqa_equals_materialised_mha():
    g = attn_inputs.paged_problem(seed=27, q_lens=[260], kv_lens=[300], num_q_heads=8,
                                  num_kv_heads=2, head_size=128, block_size=64, causal=True)
    m = attn_inputs.paged_problem(seed=27, q_lens=[260], kv_lens=[300], num_q_heads=8,
                                  num_kv_heads=8, head_size=128, block_size=64, causal=True)
    m.q = g.q.clone()
    m.k_cache = g.k_cache.repeat_interleave(4, dim=2).contiguous()
    m.v_cache = g.v_cache.repeat_interleave(4, dim=2).contiguous()
    m.block_table = g.block_table.clone()
    a, b = gpu_prefill(g), gpu_prefill(m)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_epilogue_rounding_modes(dtype):
    """The three modes must equal the oracle's rounding of the kernel's own
    unrounded fp32 result o / l (the result is deterministic)."""
    prob = attn_inputs.paged_problem(seed=28, q_lens=[300, 45], kv_lens=[300, 600], num_q_heads=4,
                                     num_kv_heads=2, head_size=128, block_size=64, dtype=dtype,
                                     causal=False, sigma=3.0)
    t = to_dev(prob)
    x = gpu_prefill(prob, t, rounding=3)
    torch.cuda.synchronize()
    xf = x.cpu().numpy().astype(np.float32)
    odt = oracle.BF16 if dtype == torch.bfloat16 else oracle.F16
    for mode in (0, 1, 2):
        r = gpu_prefill(prob, t, rounding=mode)
        torch.cuda.synchronize()
        got = r.cpu().view(torch.int16).numpy().view(np.uint16)
        exp = oracle.round_f32(xf, odt, mode)
        assert np.array_equal(got, exp), mode


def test_bad_block_table_entry_is_reported():
    prob = attn_inputs.paged_problem(seed=29, q_lens=[130], kv_lens=[300], num_q_heads=2,
                                     num_kv_heads=1, head_size=128, block_size=64, causal=True)
    prob.block_table[0, 2] = prob.num_blocks + 1000
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_prefill(prob, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5


# ----------------------------------------------------------------------------
# full-size workloads
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["prefill_causal_fp16_s128_d64", "prefill_causal_bf16_gqa_s2048",
                                  "prefill_chunked_bf16_b4"])
def test_workload_full(name):
    """The full output tensor of the 128, 2048 and chunked workloads (the
    oracle finishes them in about a second, 13 s and 52 s on 16 cores)."""
    check_full(attn_inputs.workload(name), name=name)


@pytest.mark.parametrize("name", ["prefill_causal_bf16_s8192"])
def test_workload_sampled(name):
    prob = attn_inputs.workload(name)
    out = gpu_prefill(prob)
    torch.cuda.synchronize()
    rows = sample_rows(prob, per_head_random=256)
    ref, _ = oracle_run(prob, rows=rows)
    got = as_rows(out)[rows]
    record(name + " (rows sampled)", got, ref, prob.dtype)
    err = max_err(got, ref)
    assert err <= TOL[prob.dtype], (err, worst(got, ref))


def test_workload_dense_bshd_s16384_three_roundings():
    prob = attn_inputs.workload("dense_bf16_bshd_s16384")
    t = to_dev(prob)
    rows = sample_rows(prob, per_head_random=256)
    ref, _ = oracle_run(prob, rows=rows)
    x = gpu_prefill(prob, t, rounding=3)
    torch.cuda.synchronize()
    xs = x.cpu().numpy().reshape(-1, 128)[rows].astype(np.float32)
    for mode in (0, 1, 2):
        out = gpu_prefill(prob, t, rounding=mode)
        torch.cuda.synchronize()
        got = as_rows(out)[rows]
        record(f"dense_bf16_bshd_s16384 mode {mode} (rows sampled)", got, ref, prob.dtype)
        err = max_err(got, ref)
        assert err <= TOL[prob.dtype], (mode, err, worst(got, ref))
        bits = out.cpu().view(torch.int16).numpy().reshape(-1, 128)[rows].view(np.uint16)
        assert np.array_equal(bits, oracle.round_f32(xs, oracle.BF16, mode))

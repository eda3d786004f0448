"""GPU parity of the split-KV decode and its log-sum-exp combine against the
fp64 oracle ("gfx942 unified attention, from the math up", sec. 8).

Tolerance: 4e-2 (bf16) / 2e-2 (fp16) max |err| vs the oracle, as for prefill.
Covers the full decode workload (64 sequences, kv lengths uniform in
[512, 8192], block size 16, GQA 4:1, 8 splits), every heads-per-CTA variant,
head size 64 and fp16, split counts 1..64, batches of up to 2300 sequences
(each way the kernel holds the sequence lengths), tiny and empty sequences, the
log-sum-exp output, bit identity across runs, and device-side reporting of a
bad block-table entry.
"""
import numpy as np
import pytest
import torch

import attn_inputs
from tests.helpers import (TOL, as_rows, gpu_decode, gpu_prefill, max_err, oracle_run, record,
                           to_dev, worst)

pytestmark = pytest.mark.gpu


def check(prob, splits=8, name=None, **kw):
    out = gpu_decode(prob, splits=splits, **kw)
    torch.cuda.synchronize()
    ref, _ = oracle_run(prob)
    got = as_rows(out)
    if name:
        record(name, got, ref, prob.dtype)
    err = max_err(got, ref)
    assert err <= TOL[prob.dtype], (err, worst(got, ref))
    return out


def test_workload_decode_full():
    check(attn_inputs.workload("decode_bf16_b64_paged16"), splits=8, name="decode_bf16_b64_paged16")


@pytest.mark.parametrize("name", ["decode_bf16_b64_paged16_d64", "decode_bf16_b64_paged16_d256"])
def test_workload_decode_other_head_sizes(name):
    check(attn_inputs.workload(name), splits=8, name=name)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (8, 2), (16, 2), (24, 2), (12, 4), (16, 1),
                                     (32, 1), (40, 2), (48, 1), (64, 4), (2, 1)])
def test_head_groups(hq, hkv):
    prob = attn_inputs.paged_problem(seed=31, q_lens=[1] * 5, kv_lens=[1, 16, 17, 300, 2049],
                                     num_q_heads=hq, num_kv_heads=hkv, head_size=128,
                                     block_size=16, causal=False, pool_extra=4)
    check(prob)


# The persistent kernel orders work items longest sequence first when the
# batch is small enough to rank in shared memory, keeps the sequence lengths
# in shared memory for larger batches, and reads them from global memory
# beyond that (the thresholds differ by head size); each regime, on both
# sides of its threshold, must give the same results.
@pytest.mark.parametrize("d,n,splits", [(128, 128, 8), (128, 129, 8), (128, 700, 3),
                                        (128, 2048, 8), (128, 2049, 1), (128, 2300, 8),
                                        (64, 2100, 8), (256, 1024, 8), (256, 1025, 2),
                                        (256, 1300, 8)])
def test_many_sequences(d, n, splits):
    rng = np.random.default_rng(n + d)
    kv_lens = [int(x) for x in rng.integers(0, 90, size=n)]
    kv_lens[n // 2] = 700                               # one long sequence in the middle
    prob = attn_inputs.paged_problem(seed=35 + n, q_lens=[1] * n, kv_lens=kv_lens, num_q_heads=8,
                                     num_kv_heads=2, head_size=d, block_size=16, causal=False,
                                     pool_extra=2)
    check(prob, splits=splits)


@pytest.mark.parametrize("splits", [1, 2, 3, 8, 64])
@pytest.mark.parametrize("bs", [16, 32, 256])
def test_split_counts(splits, bs):
    prob = attn_inputs.paged_problem(seed=32, q_lens=[1] * 4, kv_lens=[5, 64, 1000, 4097],
                                     num_q_heads=8, num_kv_heads=2, head_size=128, block_size=bs,
                                     causal=False)
    check(prob, splits=splits)


@pytest.mark.parametrize("splits", [1, 8])
def test_fp16_d128(splits):
    prob = attn_inputs.paged_problem(seed=38, q_lens=[1] * 3, kv_lens=[130, 9, 2500],
                                     num_q_heads=16, num_kv_heads=4, head_size=128, block_size=16,
                                     dtype=torch.float16, causal=False, sigma=2.0)
    check(prob, splits=splits)


def test_fp32_output_and_rounding_modes():
    prob = attn_inputs.paged_problem(seed=39, q_lens=[1] * 6, kv_lens=[100, 2000, 33, 700, 1, 4000],
                                     num_q_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                                     causal=False)
    from oracle import oracle
    t = to_dev(prob)
    for splits in (1, 8):
        x = gpu_decode(prob, t, splits=splits, rounding=3)
        torch.cuda.synchronize()
        xf = x.cpu().numpy().astype(np.float32)
        for mode in (0, 1, 2):
            r = gpu_decode(prob, t, splits=splits, rounding=mode)
            torch.cuda.synchronize()
            got = r.cpu().view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(got, oracle.round_f32(xf, oracle.BF16, mode)), (splits, mode)


def test_fp16_d64():
    prob = attn_inputs.paged_problem(seed=33, q_lens=[1] * 6, kv_lens=[3, 15, 16, 100, 777, 3000],
                                     num_q_heads=4, num_kv_heads=1, head_size=64, block_size=16,
                                     dtype=torch.float16, causal=False)
    check(prob)


def test_empty_sequence_and_lse():
    prob = attn_inputs.paged_problem(seed=34, q_lens=[1] * 3, kv_lens=[0, 40, 2000], num_q_heads=8,
                                     num_kv_heads=2, head_size=128, block_size=16, causal=False)
    out, lse = gpu_decode(prob, lse=True)
    torch.cuda.synchronize()
    ref, ref_lse = oracle_run(prob)
    got = as_rows(out)
    assert max_err(got, ref) <= TOL[prob.dtype]
    lh = lse.cpu().numpy().reshape(-1).astype(np.float64)
    assert np.all(np.isneginf(lh[:8])) and np.all(got[:8] == 0)
    assert np.max(np.abs(lh[8:] - ref_lse[8:])) < 2e-3


def test_decode_matches_single_row_prefill():
    prob = attn_inputs.paged_problem(seed=35, q_lens=[1] * 4, kv_lens=[129, 7, 640, 1500],
                                     num_q_heads=8, num_kv_heads=2, head_size=128, block_size=64,
                                     causal=True)
    t = to_dev(prob)
    a = gpu_decode(prob, t, splits=4)
    b = gpu_prefill(prob, t)
    torch.cuda.synchronize()
    assert (a.float() - b.float()).abs().max().item() <= 2 * TOL[prob.dtype]


def test_run_to_run_bit_identical():
    prob = attn_inputs.paged_problem(seed=36, q_lens=[1] * 16, kv_lens=list(range(100, 4100, 250)),
                                     num_q_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                                     causal=False)
    t = to_dev(prob)
    a = gpu_decode(prob, t)
    b = gpu_decode(prob, t)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_bad_block_table_entry_is_reported():
    prob = attn_inputs.paged_problem(seed=37, q_lens=[1, 1], kv_lens=[100, 100], num_q_heads=4,
                                     num_kv_heads=1, head_size=128, block_size=16, causal=False)
    prob.block_table[1, 3] = -7
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_decode(prob, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5

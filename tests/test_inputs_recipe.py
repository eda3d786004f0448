"""The seeded input generator (attn_inputs.py), which both the oracle and the
CUDA path read (CPU): the workloads have the stated shapes and length mix,
the paged layout is a valid one (every page owned by at most one sequence,
unused table entries -1, slots past a sequence's end poisoned with NaN so
that a kernel reading them would show), and the draws are reproducible
from the seed."""
import math

import numpy as np
import pytest
import torch

import attn_inputs


def check_layout(prob):
    bt = prob.block_table.numpy()
    n_blocks = prob.k_cache.shape[0]
    bs = prob.block_size
    seen = set()
    for b, sk in enumerate(prob.kv_lens):
        npg = -(-sk // bs)
        ids = bt[b, :npg]
        assert (ids >= 0).all() and (ids < n_blocks).all()
        assert (bt[b, npg:] == -1).all()
        for i in ids:
            assert int(i) not in seen            # no page shared between sequences
            seen.add(int(i))
        k = prob.k_cache[torch.as_tensor(ids, dtype=torch.long)].float().reshape(npg * bs, -1)
        assert torch.isfinite(k[:sk]).all()      # the sequence's keys are real draws
        assert torch.isnan(k[sk:]).all()         # the rest of its last page is poison
    qsl = prob.query_start_loc.numpy()
    assert qsl[0] == 0 and (np.diff(qsl) == np.array(prob.q_lens)).all()
    assert (prob.seq_lens.numpy() == np.array(prob.kv_lens)).all()


def test_small_problem_layout_and_reproducibility():
    kw = dict(q_lens=[5, 0, 40], kv_lens=[70, 3, 40], num_q_heads=4, num_kv_heads=2,
              head_size=64, block_size=16, pool_extra=3)
    a = attn_inputs.paged_problem(seed=3, **kw)
    check_layout(a)
    assert a.k_cache.shape[0] == 5 + 1 + 3 + 3   # pages used + unreferenced extras
    b = attn_inputs.paged_problem(seed=3, **kw)
    for name in ("q", "k_cache", "v_cache", "block_table"):
        x, y = getattr(a, name), getattr(b, name)
        assert torch.equal(x.view(torch.int16) if x.dtype.is_floating_point else x,
                           y.view(torch.int16) if y.dtype.is_floating_point else y)
    c = attn_inputs.paged_problem(seed=4, **kw)
    assert not torch.equal(a.q, c.q)
    assert a.scale == 1.0 / 8.0


def test_value_draws_do_not_depend_on_the_page_order():
    """The layout and the values come from separate generators, so the same
    seed with and without a permuted table gives the same keys in order."""
    kw = dict(q_lens=[3, 9], kv_lens=[50, 33], num_q_heads=2, num_kv_heads=1, head_size=64,
              block_size=16)
    p = attn_inputs.paged_problem(seed=8, permute=True, **kw)
    u = attn_inputs.paged_problem(seed=8, permute=False, **kw)

    def dense_keys(prob, b):
        ids = prob.block_table[b, :-(-prob.kv_lens[b] // 16)].long()
        return prob.k_cache[ids].reshape(-1, 64)[:prob.kv_lens[b]]

    for b in range(2):
        assert torch.equal(dense_keys(p, b).view(torch.int16), dense_keys(u, b).view(torch.int16))
    assert torch.equal(p.q.view(torch.int16), u.q.view(torch.int16))


def test_fp8_caches_hold_scaled_codes():
    prob = attn_inputs.paged_problem(seed=5, q_lens=[4], kv_lens=[300], num_q_heads=4,
                                     num_kv_heads=2, head_size=128, block_size=64, sigma=1.0,
                                     kv_dtype=torch.float8_e4m3fn)
    assert prob.kv_fp8 and prob.k_cache.dtype == torch.float8_e4m3fn
    assert prob.k_scale == prob.v_scale == pytest.approx(6.0 / 448.0)
    k = prob.k_cache.float()
    fin = k[torch.isfinite(k)]
    assert fin.abs().max() <= 448.0
    # +-6 sigma spans the format: the scaled draws have unit spread
    assert 0.8 < float((fin * prob.k_scale).std()) < 1.2
    check_layout(prob)


@pytest.mark.parametrize("name,shape", [
    ("prefill_causal_fp16_s128_d64", (1, 2, 2, 64, 128, torch.float16)),
    ("prefill_causal_bf16_gqa_s2048", (1, 32, 8, 128, 64, torch.bfloat16)),
    ("prefill_chunked_bf16_b4", (4, 32, 8, 128, 64, torch.bfloat16)),
])
def test_prefill_workload_shapes(name, shape):
    b, hq, hkv, d, bs, dtype = shape
    prob = attn_inputs.workload(name)
    assert (prob.num_seqs, prob.num_q_heads, prob.num_kv_heads, prob.head_size,
            prob.block_size, prob.dtype) == shape
    assert prob.causal
    check_layout(prob)


def test_decode_workload_length_mix():
    prob = attn_inputs.workload("decode_bf16_b64_paged16")
    assert (prob.num_seqs, prob.num_q_heads, prob.num_kv_heads, prob.head_size,
            prob.block_size) == (64, 32, 8, 128, 16)
    assert prob.q_lens == [1] * 64 and not prob.causal
    lens = np.array(prob.kv_lens)
    assert lens.min() >= 512 and lens.max() <= 8192
    # uniform on [512, 8192]: mean 4352, sd 2217; 64 draws land within 4 s.e.
    assert abs(lens.mean() - 4352) < 4 * 2217 / math.sqrt(64)
    assert len(set(lens.tolist())) > 50
    check_layout(prob)
    assert attn_inputs.random_kv_lens(0, 64, 512, 8192) == prob.kv_lens
    assert attn_inputs.random_kv_lens(1, 64, 512, 8192) != prob.kv_lens

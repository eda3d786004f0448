"""GPU parity of attn_fwd_prefill_split (the persistent grid that cuts the key
range of units across CTAs and merges the parts by the log-sum-exp combine of
"gfx942 unified attention, from the math up", sec. 8) against the fp64
oracle.

Tolerance: 2e-2 (fp16) / 4e-2 (bf16) max |err|, the gate of sec. 10, and the
log-sum-exp within 2e-3.  The split path sums a cut unit's keys in parts, so
it is compared with the one-shot call within that tolerance, not bit for
bit; it must be bit-identical from run to run and must not depend on what an
earlier call (or nothing) left in its workspace.
"""
import numpy as np
import pytest
import torch

import attn_inputs
from tests.helpers import (TOL, as_rows, gpu_prefill, max_err, oracle_run, record, sample_rows,
                           to_dev, worst)

pytestmark = pytest.mark.gpu


def split_prefill(prob, t=None, rounding=0, lse=False, workspace=None):
    import attention_forward_sdpa_gb300 as attn
    t = t or to_dev(prob)
    out = torch.empty(t["q"].shape, dtype=torch.float32 if rounding == 3 else t["q"].dtype,
                      device="cuda")
    lse_t = torch.empty(t["q"].shape[:2], dtype=torch.float32, device="cuda") if lse else None
    ws = workspace
    if ws is None:
        ws = torch.empty(attn.attn_prefill_split_workspace_size(prob.head_size), dtype=torch.uint8,
                         device="cuda")
    attn.attn_fwd_prefill(out, t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                          t["query_start_loc"], t["seq_lens"], max_seqlen_q=prob.max_seqlen_q,
                          max_seqlen_k=prob.max_seqlen_k, scale=prob.scale, causal=prob.causal,
                          rounding=rounding, lse=lse_t, split_workspace=ws)
    return (out, lse_t) if lse else out


def check(prob, got, rows=None, name=None, lse=None):
    torch.cuda.synchronize()
    ref, ref_lse = oracle_run(prob, rows=rows)
    g = as_rows(got)
    if rows is not None:
        g = g[rows]
    if name:
        record(name, g, ref, prob.dtype)
    err = max_err(g, ref)
    assert err <= TOL[prob.dtype], (err, worst(g, ref))
    if lse is not None:
        gl = lse.cpu().numpy().reshape(-1).astype(np.float64)
        if rows is not None:
            gl = gl[rows]
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(gl), fin)
        if fin.any():
            assert np.max(np.abs(gl[fin] - ref_lse[fin])) < 2e-3


@pytest.mark.parametrize("name", ["prefill_causal_bf16_gqa_s2048", "prefill_chunked_bf16_b4"])
def test_split_workload_full_tensor(name):
    prob = attn_inputs.workload(name)
    t = to_dev(prob)
    out, lse = split_prefill(prob, t, lse=True)
    check(prob, out, name=name + " (split)", lse=lse)
    # run-to-run bit identity, and the one-shot kernel within the tolerance
    again = split_prefill(prob, t)
    torch.cuda.synchronize()
    assert torch.equal(out, again)
    one = gpu_prefill(prob, t)
    torch.cuda.synchronize()
    d = (one.float() - out.float()).abs().max().item()
    assert d <= TOL[prob.dtype], d


@pytest.mark.parametrize("name,rounding", [("prefill_causal_bf16_s8192", 0),
                                           ("dense_bf16_bshd_s16384", 2)])
def test_split_workload_rows_sampled(name, rounding):
    prob = attn_inputs.workload(name)
    out = split_prefill(prob, rounding=rounding)
    rows = sample_rows(prob, per_head_random=16)
    torch.cuda.synchronize()
    ref, _ = oracle_run(prob, rows=rows)
    g = as_rows(out)[rows]
    record(f"{name} mode {rounding} (split, rows sampled)", g, ref, prob.dtype)
    err = max_err(g, ref)
    assert err <= TOL[prob.dtype], (err, worst(g, ref))


SMALL = {
    # ragged batch, GQA 4:1 (head pairs), block 64, causal
    "gqa4_bf16_d128_varlen_causal": dict(q_lens=[300, 1, 129, 77, 640], kv_lens=[300, 500, 129, 1000, 700],
                                         num_q_heads=8, num_kv_heads=2, head_size=128, block_size=64,
                                         dtype=torch.bfloat16, causal=True),
    # non-causal, fp16, block 16
    "gqa2_fp16_d128_noncausal": dict(q_lens=[450, 200], kv_lens=[700, 333], num_q_heads=4,
                                     num_kv_heads=2, head_size=128, block_size=16,
                                     dtype=torch.float16, causal=False),
    # odd group (two row blocks of one head per unit), head size 64, block 128
    "gqa3_bf16_d64_causal": dict(q_lens=[900, 130], kv_lens=[900, 400], num_q_heads=6,
                                 num_kv_heads=2, head_size=64, block_size=128,
                                 dtype=torch.bfloat16, causal=True),
    # rows that see no key (Sq > Sk, causal) and an empty KV sequence
    "zero_rows": dict(q_lens=[600, 300, 50], kv_lens=[200, 0, 900], num_q_heads=4, num_kv_heads=2,
                      head_size=128, block_size=32, dtype=torch.bfloat16, causal=True),
    # MHA, many sequences of one row block
    "mha_bf16_many": dict(q_lens=[128] * 40, kv_lens=[128 + 37 * i for i in range(40)],
                          num_q_heads=2, num_kv_heads=2, head_size=128, block_size=64,
                          dtype=torch.bfloat16, causal=True),
}


@pytest.mark.parametrize("case", sorted(SMALL))
def test_split_small_cases(case):
    prob = attn_inputs.paged_problem(seed=31, **SMALL[case])
    out, lse = split_prefill(prob, lse=True)
    check(prob, out, lse=lse)


@pytest.mark.parametrize("rounding", [1, 3])
def test_split_roundings(rounding):
    prob = attn_inputs.paged_problem(seed=32, **SMALL["gqa4_bf16_d128_varlen_causal"])
    out = split_prefill(prob, rounding=rounding)
    check(prob, out)


def test_split_workspace_reuse_and_garbage():
    """Calls in a row on one workspace, different problems, then a workspace
    full of arbitrary bytes: each result matches the oracle."""
    import attention_forward_sdpa_gb300 as attn
    ws = torch.empty(attn.attn_prefill_split_workspace_size(128), dtype=torch.uint8, device="cuda")
    probs = [attn_inputs.paged_problem(seed=40 + i, **SMALL[c])
             for i, c in enumerate(["gqa4_bf16_d128_varlen_causal", "mha_bf16_many",
                                    "gqa4_bf16_d128_varlen_causal"])]
    for prob in probs:
        check(prob, split_prefill(prob, workspace=ws))
    ws.fill_(0xFF)
    check(probs[0], split_prefill(probs[0], workspace=ws))
    ws.random_(0, 256)
    check(probs[1], split_prefill(probs[1], workspace=ws))


def test_split_rejects_a_missing_or_short_workspace():
    import attention_forward_sdpa_gb300 as attn
    prob = attn_inputs.paged_problem(seed=33, **SMALL["mha_bf16_many"])
    short = torch.empty(attn.attn_prefill_split_workspace_size(128) - 256, dtype=torch.uint8,
                        device="cuda")
    with pytest.raises(attn.AttnError) as e:
        split_prefill(prob, workspace=short)
    assert e.value.status == 4

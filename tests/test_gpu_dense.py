"""GPU parity of the strided dense entry point (attn_fwd_dense): fixed-length
batches read in place from BSHD [B, S, H, d] or BHSD [B, H, S, d] memory.

The seeded generator with block_size = Sk and an unpermuted table lays the K/V
cache out exactly as a dense BSHD batch, so the same problem feeds the fp64
oracle (tolerance 2e-2 fp16 / 4e-2 bf16 max |err|, as for the paged path) and
the paged GPU path, which the dense path must reproduce bit for bit (same
arithmetic, only the addressing differs).
"""
import numpy as np
import pytest
import torch

import attn_inputs
from tests.helpers import TOL, as_rows, gpu_prefill, max_err, oracle_run, sample_rows, worst

pytestmark = pytest.mark.gpu


def make(B, Sq, Sk, Hq, Hkv, d, dtype, causal, seed=0, sigma=1.0):
    return attn_inputs.paged_problem(seed=seed, q_lens=[Sq] * B, kv_lens=[Sk] * B,
                                     num_q_heads=Hq, num_kv_heads=Hkv, head_size=d,
                                     block_size=Sk, dtype=dtype, causal=causal, permute=False,
                                     poison=False, sigma=sigma)


def dense_tensors(prob, B, Sq, Sk, layout, pad=0):
    """Device tensors in the requested memory layout (pad > 0: each head row is
    padded by `pad` elements, so that no stride is the dense one)."""
    Hq, Hkv, d = prob.num_q_heads, prob.num_kv_heads, prob.head_size
    out = []
    for x, S, H in ((prob.q.view(B, Sq, Hq, d), Sq, Hq), (prob.k_cache.view(B, Sk, Hkv, d), Sk, Hkv),
                    (prob.v_cache.view(B, Sk, Hkv, d), Sk, Hkv)):
        x = x.cuda()
        if layout == "bhsd":
            x = x.transpose(1, 2)                       # [B, H, S, d] view
        if pad:
            big = torch.zeros(*x.shape[:3], d + pad, dtype=x.dtype, device="cuda")
            big[..., :d] = x
            x = big[..., :d]
        else:
            x = x.contiguous()
        out.append(x)
    return out


def run_dense(prob, B, Sq, Sk, layout, rounding=0, lse=False, pad=0):
    import attention_forward_sdpa_gb300 as attn
    q, k, v = dense_tensors(prob, B, Sq, Sk, layout, pad)
    res = attn.dense(q, k, v, layout=layout, scale=prob.scale, causal=prob.causal,
                     rounding=rounding, return_lse=lse)
    out = res[0] if lse else res
    packed = (out if layout == "bshd" else out.transpose(1, 2)).contiguous()
    packed = packed.view(B * Sq, prob.num_q_heads, prob.head_size)
    if lse:
        return packed, res[1]                            # lse: [B, Hq, Sq]
    return packed


CASES = {
    "gqa4_bf16_d128_causal_ragged": (2, 200, 333, 8, 2, 128, torch.bfloat16, True),
    "mha_fp16_d64_noncausal": (2, 256, 384, 4, 4, 64, torch.float16, False),
    "gqa3_bf16_d128_causal_rows_without_keys": (1, 300, 130, 6, 2, 128, torch.bfloat16, True),
    "gqa2_bf16_d128_noncausal_short_keys": (3, 129, 17, 4, 2, 128, torch.bfloat16, False),
    "mha_bf16_d128_causal_square": (2, 384, 384, 2, 2, 128, torch.bfloat16, True),
    "gqa8_fp16_d128_causal": (1, 257, 512, 16, 2, 128, torch.float16, True),
    "gqa2_bf16_d128_causal_many_batches": (600, 24, 40, 4, 2, 128, torch.bfloat16, True),
}


@pytest.mark.parametrize("layout", ["bshd", "bhsd"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_dense_matches_oracle(name, layout):
    B, Sq, Sk, Hq, Hkv, d, dtype, causal = CASES[name]
    prob = make(B, Sq, Sk, Hq, Hkv, d, dtype, causal)
    out = run_dense(prob, B, Sq, Sk, layout)
    torch.cuda.synchronize()
    ref, _ = oracle_run(prob)
    got = as_rows(out)
    err = max_err(got, ref)
    assert err <= TOL[dtype], (err, worst(got, ref))


@pytest.mark.parametrize("layout", ["bshd", "bhsd"])
def test_dense_padded_strides(layout):
    prob = make(2, 160, 256, 4, 2, 128, torch.bfloat16, True, seed=3)
    out = run_dense(prob, 2, 160, 256, layout, pad=8)
    torch.cuda.synchronize()
    ref, _ = oracle_run(prob)
    assert max_err(as_rows(out), ref) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("layout", ["bshd", "bhsd"])
@pytest.mark.parametrize("causal", [True, False])
def test_dense_equals_paged_bitwise(layout, causal):
    """Sk a multiple of 128 so that the paged entry point accepts block_size = Sk."""
    B, Sq, Sk, Hq, Hkv = 2, 256, 384, 8, 2
    prob = make(B, Sq, Sk, Hq, Hkv, 128, torch.bfloat16, causal, seed=5)
    out, lse = run_dense(prob, B, Sq, Sk, layout, lse=True)
    ref_out, ref_lse = gpu_prefill(prob, lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    # paged LSE is [total_q, Hq]; dense is [B, Hq, Sq]
    assert torch.equal(lse, ref_lse.view(B, Sq, Hq).transpose(1, 2))


@pytest.mark.parametrize("rounding", [1, 2, 3])
def test_dense_roundings_bhsd(rounding):
    B, Sq, Sk = 2, 200, 256
    prob = make(B, Sq, Sk, 4, 2, 128, torch.bfloat16, False, seed=7)
    out = run_dense(prob, B, Sq, Sk, "bhsd", rounding=rounding)
    ref_paged = gpu_prefill(prob, rounding=rounding)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_paged)
    ref, _ = oracle_run(prob)
    assert max_err(as_rows(out), ref) <= TOL[torch.bfloat16]


def test_dense_bhsd_full_size_sampled():
    """The dense workload (B=4, H=16, S=16384, d=128, non-causal bf16) read in
    BHSD memory, RTZ output; sampled rows against the oracle."""
    prob = attn_inputs.workload("dense_bf16_bshd_s16384")
    B, S = 4, 16384
    out = run_dense(prob, B, S, S, "bhsd", rounding=2)
    torch.cuda.synchronize()
    rows = sample_rows(prob, per_head_random=2)
    ref, _ = oracle_run(prob, rows=rows)
    got = as_rows(out)[rows]
    err = max_err(got, ref)
    assert err <= TOL[torch.bfloat16], (err, worst(got, ref))

"""Pins of the oracle's fp8 K/V reading (CPU only).

"gfx942 unified attention, from the math up" sec. 9 lists fp8 K/V among the
feature flags without defining it; the oracle takes the common convention
(stated in oracle/sdpa_oracle.c): the caches hold OCP E4M3 codes and the key
and value meant are the widened code times a per-tensor factor.  The pins:
  - the E4M3 widening against torch's float8_e4m3fn -> float64 conversion on
    all 256 patterns (library routine), and against values fixed by the
    format's definition (largest finite 448, smallest subnormal 2^-9,
    smallest normal 2^-6, 1.0, signed zero, the two NaN codes);
  - every E4M3 value is a bf16 value, so with unit factors an fp8 problem must
    equal, bit for bit in binary64, the bf16 problem holding the same values:
    this ties the 1-byte addressing and layout to the 16-bit path;
  - the factors act on the right tensors: K's factor is a factor on the
    scores (equal to scaling tau), V's a factor on the output;
  - a library cross-check: torch float64 SDPA on the dequantised logical K/V.
"""
import math

import numpy as np
import pytest
import torch

import attn_inputs
from oracle import oracle
from tests.test_oracle_pins import dense_logical

F8 = torch.float8_e4m3fn


def test_widen8_matches_torch_on_all_patterns():
    bits = np.arange(256, dtype=np.uint8)
    got = oracle.widen8(bits)
    ref = torch.from_numpy(bits.copy()).view(F8).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(ref[fin]))


def test_widen8_fixed_points():
    w = oracle.widen8(np.array([0x7E, 0x01, 0x08, 0x38, 0x80, 0x00, 0x7F, 0xFF, 0xFE, 0x07],
                               dtype=np.uint8))
    assert w[0] == 448.0
    assert w[1] == 2.0 ** -9
    assert w[2] == 2.0 ** -6
    assert w[3] == 1.0
    assert w[4] == 0.0 and math.copysign(1.0, w[4]) < 0
    assert w[5] == 0.0 and math.copysign(1.0, w[5]) > 0
    assert np.isnan(w[6]) and np.isnan(w[7])
    assert w[8] == -448.0
    assert w[9] == 7 * 2.0 ** -9          # largest subnormal, 0.875 * 2^-6


def fp8_problem(seed, causal=True, hq=4, hkv=2, d=32, bs=16, q_lens=(7, 1, 12),
                kv_lens=(19, 40, 12)):
    return attn_inputs.paged_problem(seed=seed, q_lens=list(q_lens), kv_lens=list(kv_lens),
                                     num_q_heads=hq, num_kv_heads=hkv, head_size=d,
                                     block_size=bs, causal=causal, kv_dtype=F8, pool_extra=2)


def run(prob, scale=None, k_scale=None, v_scale=None, kv16=None, dtype=oracle.BF16):
    k, v = (prob.k_cache, prob.v_cache) if kv16 is None else kv16
    scales = None if kv16 is not None else (prob.k_scale if k_scale is None else k_scale,
                                             prob.v_scale if v_scale is None else v_scale)
    return oracle.sdpa(prob.q, k, v, prob.block_table, prob.query_start_loc, prob.seq_lens,
                       num_q_heads=prob.num_q_heads, num_kv_heads=prob.num_kv_heads,
                       head_size=prob.head_size, block_size=prob.block_size,
                       scale=prob.scale if scale is None else scale, causal=prob.causal,
                       dtype=dtype, n_threads=4, kv_scales=scales)


@pytest.mark.parametrize("causal", [True, False])
def test_unit_factor_fp8_equals_bf16_holding_the_same_values(causal):
    prob = fp8_problem(11, causal=causal)
    # E4M3 -> bf16 is exact (3 fraction bits, exponents 2^-9 .. 2^8), NaN stays NaN
    k16 = prob.k_cache.to(torch.float32).to(torch.bfloat16)
    v16 = prob.v_cache.to(torch.float32).to(torch.bfloat16)
    assert torch.equal(k16.to(torch.float32).nan_to_num(7.0),
                       prob.k_cache.to(torch.float32).nan_to_num(7.0))
    o8, l8 = run(prob, k_scale=1.0, v_scale=1.0)
    o16, l16 = run(prob, kv16=(k16, v16))
    assert np.array_equal(o8, o16)
    assert np.array_equal(l8, l16)


def test_k_factor_scales_the_scores_and_v_factor_the_output():
    prob = fp8_problem(12)
    # factors near the generator's own (codes are ~N(0, 75^2)), so scores stay O(1)
    a, b = prob.k_scale * 0.9, prob.v_scale * 3.0
    o, lse = run(prob, k_scale=a, v_scale=b)
    o1, lse1 = run(prob, scale=prob.scale * a, k_scale=1.0, v_scale=1.0)
    assert np.max(np.abs(o - b * o1)) < 1e-12 * max(1.0, np.max(np.abs(o)))
    fin = np.isfinite(lse1)
    assert np.max(np.abs(lse[fin] - lse1[fin])) < 1e-12
    # swapping the two factors gives a different answer (the pin can fail)
    o_sw, _ = run(prob, k_scale=b, v_scale=a)
    assert np.max(np.abs(o_sw - o)) > 1e-3


@pytest.mark.parametrize("causal", [True, False])
def test_fp8_matches_torch_sdpa_on_dequantised_values(causal):
    prob = fp8_problem(13, causal=causal, hq=6, hkv=3)
    got, _ = run(prob)
    g = prob.num_q_heads // prob.num_kv_heads
    row = 0
    for b in range(prob.num_seqs):
        q0, q1 = int(prob.query_start_loc[b]), int(prob.query_start_loc[b + 1])
        sq, sk = q1 - q0, prob.kv_lens[b]
        q = prob.q[q0:q1].to(torch.float64).permute(1, 0, 2)             # [H, Sq, d]
        k, v = dense_logical(prob, b)                                    # E4M3 -> float64
        k = (k * prob.k_scale).permute(1, 0, 2).repeat_interleave(g, dim=0)
        v = (v * prob.v_scale).permute(1, 0, 2).repeat_interleave(g, dim=0)
        mask = torch.ones(sq, sk, dtype=torch.bool).tril(diagonal=sk - sq) if causal else None
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask,
                                                               scale=prob.scale)
        ref = ref.permute(1, 0, 2).reshape(-1, prob.head_size).numpy()
        n = sq * prob.num_q_heads
        assert np.max(np.abs(got[row:row + n] - ref)) < 1e-12
        row += n

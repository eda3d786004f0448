"""Pins of the oracle's feature-flagged variants (CPU only).

"gfx942 unified attention, from the math up" sec. 9 names sinks, ALiBi,
softcap and sliding window as feature flags without defining them; the
oracle takes their usual definitions (stated in oracle/sdpa_oracle.c).  Each
test ties one of them to something other than the oracle's own formula:
  - limits in which the feature disappears (an unbounded window, a cap or a
    sink far away, a zero slope) must give the plain definition exactly;
  - limits with closed forms: a zero-width window or an overwhelming ALiBi
    slope leaves only the aligned key (O = V of that key), a vanishing cap
    makes every score 0 (O = mean of the visible values), saturated scores
    take the values +-cap, a dominant sink drives O to 0;
  - a geometric-series closed form for ALiBi weights with a zero query, and
    the closed form sum(V) / (n + e^z) for a sink with a zero query;
  - a library cross-check of the window's orientation (torch float64 SDPA
    with an independently built band mask).
"""
import math

import numpy as np
import pytest
import torch

import attn_inputs
from oracle import oracle
from tests.test_oracle_pins import dense_logical


def run(prob, **feat):
    return oracle.sdpa(prob.q, prob.k_cache, prob.v_cache, prob.block_table,
                       prob.query_start_loc, prob.seq_lens,
                       num_q_heads=prob.num_q_heads, num_kv_heads=prob.num_kv_heads,
                       head_size=prob.head_size, block_size=prob.block_size,
                       scale=prob.scale, causal=prob.causal,
                       dtype=oracle.BF16 if prob.dtype == torch.bfloat16 else oracle.F16,
                       n_threads=4, **feat)


def problem(seed, causal=True, q_lens=(6, 1, 9), kv_lens=(11, 7, 9), hq=4, hkv=2, d=16, **kw):
    return attn_inputs.paged_problem(seed=seed, q_lens=list(q_lens), kv_lens=list(kv_lens),
                                     num_q_heads=hq, num_kv_heads=hkv, head_size=d, block_size=4,
                                     causal=causal, pool_extra=2, **kw)


def rows_of(prob):
    """(row id, sequence, query index i, diag = i + Sk - Sq, head) for every row."""
    out = []
    for b in range(prob.num_seqs):
        q0, q1 = int(prob.query_start_loc[b]), int(prob.query_start_loc[b + 1])
        sq, sk = q1 - q0, prob.kv_lens[b]
        for i in range(sq):
            for h in range(prob.num_q_heads):
                out.append(((q0 + i) * prob.num_q_heads + h, b, i, i + sk - sq, h))
    return out


# ---------------------------------------------------------------- sliding window

@pytest.mark.parametrize("causal", [True, False])
def test_unbounded_window_is_plain(causal):
    prob = problem(40, causal)
    ref, ref_lse = run(prob)
    out, lse = run(prob, window=(1000, 1000))
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)


@pytest.mark.parametrize("causal", [True, False])
def test_zero_width_window_is_the_aligned_value_row(causal):
    prob = problem(41, causal, q_lens=(6, 9, 3), kv_lens=(11, 7, 9))
    out, lse = run(prob, window=(0, 0))
    g = prob.num_q_heads // prob.num_kv_heads
    for rid, b, i, diag, h in rows_of(prob):
        if 0 <= diag < prob.kv_lens[b]:
            _, v = dense_logical(prob, b)
            assert np.array_equal(out[rid], v[diag, h // g].numpy())
        else:                                   # the aligned key does not exist
            assert np.all(out[rid] == 0) and lse[rid] == -np.inf


@pytest.mark.parametrize("left,right", [(3, -1), (0, 2), (2, 5), (5, 0)])
def test_window_matches_torch_band_mask(left, right):
    """Library cross-check (non-causal, so that both bounds act): torch's
    float64 SDPA with the boolean band mask diag - left <= j <= diag + right."""
    prob = problem(42, causal=False, q_lens=(7, 4), kv_lens=(12, 10))
    out, _ = run(prob, window=(left, right))
    g = prob.num_q_heads // prob.num_kv_heads
    for b in range(prob.num_seqs):
        q0, q1 = int(prob.query_start_loc[b]), int(prob.query_start_loc[b + 1])
        sq, sk = q1 - q0, prob.kv_lens[b]
        q = prob.q[q0:q1].to(torch.float64).permute(1, 0, 2)
        k, v = dense_logical(prob, b)
        k = k.permute(1, 0, 2).repeat_interleave(g, dim=0)
        v = v.permute(1, 0, 2).repeat_interleave(g, dim=0)
        i = torch.arange(sq).view(-1, 1) + (sk - sq)
        j = torch.arange(sk).view(1, -1)
        mask = torch.ones(sq, sk, dtype=torch.bool)
        if left >= 0:
            mask &= j >= i - left
        if right >= 0:
            mask &= j <= i + right
        o = torch.nn.functional.scaled_dot_product_attention(
            q.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0), attn_mask=mask, scale=prob.scale)
        ref = o[0].permute(1, 0, 2).reshape(sq * prob.num_q_heads, -1).numpy()
        got = out[q0 * prob.num_q_heads:q1 * prob.num_q_heads]
        assert np.max(np.abs(got - ref)) < 1e-12


# ---------------------------------------------------------------- softcap

@pytest.mark.parametrize("causal", [True, False])
def test_distant_softcap_is_plain(causal):
    prob = problem(43, causal)
    ref, ref_lse = run(prob)
    out, lse = run(prob, softcap=1e9)
    assert np.max(np.abs(out - ref)) < 1e-12 and np.max(np.abs(lse - ref_lse)) < 1e-12


def test_vanishing_softcap_gives_the_mean_of_visible_values():
    prob = problem(44, True)
    out, _ = run(prob, softcap=1e-15)
    g = prob.num_q_heads // prob.num_kv_heads
    for rid, b, i, diag, h in rows_of(prob):
        _, v = dense_logical(prob, b)
        assert np.max(np.abs(out[rid] - v[:diag + 1, h // g].mean(0).numpy())) < 1e-12


def test_saturated_scores_take_plus_minus_cap():
    """With |tau q.k| >> cap every capped score is +cap or -cap, so the
    weights are e^(+-cap) by the sign of the raw score."""
    prob = problem(45, False, q_lens=(3,), kv_lens=(10,), hq=2, hkv=2, d=8, sigma=1.0,
                   poison=False)
    # keys +-e_0 (signs from the seeded draw), queries 4096 e_0: raw scores
    # +-4096 tau, all exact in bf16
    sign = torch.sign(prob.k_cache[..., :1]).clamp(min=-1, max=1)
    sign[sign == 0] = 1
    prob.k_cache.zero_()
    prob.k_cache[..., :1] = sign
    prob.q.zero_()
    prob.q[..., 0] = 4096.0
    cap = 2.5
    out, _ = run(prob, softcap=cap)
    k, v = dense_logical(prob, 0)
    for rid, b, i, diag, h in rows_of(prob):
        q = prob.q[i, h].to(torch.float64)
        raw = (k[:, h] @ q).numpy() * prob.scale
        assert np.min(np.abs(raw)) > 50 * cap        # tanh is 1 to fp64 precision
        w = np.exp(np.where(raw > 0, cap, -cap))
        ref = (w[:, None] * v[:, h].numpy()).sum(0) / w.sum()
        assert np.max(np.abs(out[rid] - ref)) < 1e-12


# ---------------------------------------------------------------- ALiBi

def test_zero_slopes_are_plain():
    prob = problem(46, True)
    ref, ref_lse = run(prob)
    out, lse = run(prob, alibi_slopes=np.zeros(prob.num_q_heads))
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)


@pytest.mark.parametrize("causal", [True, False])
def test_overwhelming_slope_selects_the_aligned_key(causal):
    """-a |diag - j| with a huge a leaves only j = diag (on both sides of it
    when non-causal: the bias is symmetric in the distance)."""
    prob = problem(47, causal, q_lens=(5, 4), kv_lens=(9, 4))
    out, _ = run(prob, alibi_slopes=np.full(prob.num_q_heads, 1e4))
    g = prob.num_q_heads // prob.num_kv_heads
    for rid, b, i, diag, h in rows_of(prob):
        _, v = dense_logical(prob, b)
        assert np.max(np.abs(out[rid] - v[diag, h // g].numpy())) < 1e-12


def test_alibi_geometric_weights_closed_form():
    """Zero query, causal, value channel 0 = key index j: the weights are
    r^k with r = e^-a over the distance k = diag - j, so
    O[0] = diag - sum k r^k / sum r^k, a geometric series."""
    prob = problem(48, True, q_lens=(4,), kv_lens=(20,), hq=2, hkv=1, d=8, poison=False,
                   permute=False)
    prob.q.zero_()
    for j in range(20):
        page, slot = int(prob.block_table[0, j // 4]), j % 4
        prob.v_cache[page, slot, 0, 0] = float(j)       # exact in bf16
    slopes = np.array([0.25, 1.5])
    out, _ = run(prob, alibi_slopes=slopes)
    for rid, b, i, diag, h in rows_of(prob):
        r, n = math.exp(-slopes[h]), diag + 1
        s0 = (1 - r ** n) / (1 - r)
        s1 = r * (1 - n * r ** (n - 1) + (n - 1) * r ** n) / (1 - r) ** 2
        assert abs(out[rid][0] - (diag - s1 / s0)) < 1e-12


# ---------------------------------------------------------------- sinks

def test_absent_sink_is_plain():
    prob = problem(49, True)
    ref, ref_lse = run(prob)
    out, lse = run(prob, sinks=np.full(prob.num_q_heads, -np.inf))
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)


def test_dominant_sink_drives_the_output_to_zero():
    prob = problem(50, True)
    z = 1e3
    out, lse = run(prob, sinks=np.full(prob.num_q_heads, z))
    assert np.max(np.abs(out)) < 1e-300 * 1e3 or np.max(np.abs(out)) < 1e-100
    assert np.max(np.abs(lse - z)) < 1e-12


def test_sink_with_zero_query_closed_form():
    """All scores 0, n visible keys, sink z: O = sum V / (n + e^z),
    lse = log(n + e^z)."""
    prob = problem(51, True, q_lens=(5,), kv_lens=(8,), hq=2, hkv=1)
    prob.q.zero_()
    sinks = np.array([0.0, 1.75])
    out, lse = run(prob, sinks=sinks)
    _, v = dense_logical(prob, 0)
    for rid, b, i, diag, h in rows_of(prob):
        n = diag + 1
        den = n + math.exp(sinks[h])
        assert np.max(np.abs(out[rid] - v[:n, 0].sum(0).numpy() / den)) < 1e-12
        assert abs(lse[rid] - math.log(den)) < 1e-12


def test_row_without_keys_reports_the_sink():
    prob = problem(52, True, q_lens=(6,), kv_lens=(2,), hq=2, hkv=1)
    out, lse = run(prob, sinks=np.array([0.5, -2.0]))
    for rid, b, i, diag, h in rows_of(prob):
        if diag < 0:
            assert np.all(out[rid] == 0) and lse[rid] == [0.5, -2.0][h]


def test_bad_feature_arguments_are_rejected():
    prob = problem(53, True)
    with pytest.raises(ValueError):
        run(prob, softcap=-1.0)
    with pytest.raises(ValueError):
        run(prob, window=(-2, 0))
    with pytest.raises(ValueError):
        run(prob, alibi_slopes=np.zeros(3))

"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test ties one part of the oracle to the pages or to mathematics:
  - a library routine (torch's float64 CPU scaled_dot_product_attention with an
    explicit bottom-right boolean mask; torch's bf16/fp16 casts),
  - hand-derived fixtures under tests/golden (mask orientation, rounding ties),
  - closed forms (two-key softmax, identical keys, constant scores, first
    causal row) and invariants (shift invariance, GQA as repeated K/V, paging
    and permutation invariance, convex hull),
  - brute force (nearest representable value among all 65536 patterns),
  - the exactness claims of "gfx942 unified attention, from the math up"
    sec. 3 (streaming recurrence equals the definition) and sec. 8 (split plus
    log-sum-exp combine equals the definition).
"""
import math
import os

import numpy as np
import pytest
import torch

import attn_inputs
from oracle import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run(prob, rows=None, variant=0, param=0, threads=4):
    return oracle.sdpa(prob.q, prob.k_cache, prob.v_cache, prob.block_table,
                       prob.query_start_loc, prob.seq_lens,
                       num_q_heads=prob.num_q_heads, num_kv_heads=prob.num_kv_heads,
                       head_size=prob.head_size, block_size=prob.block_size,
                       scale=prob.scale, causal=prob.causal,
                       dtype=oracle.BF16 if prob.dtype == torch.bfloat16 else oracle.F16,
                       rows=rows, variant=variant, param=param, n_threads=threads)


def dense_logical(prob, b):
    """Gathers sequence b's logical K/V [Sk, Hkv, d] as float64 (test-side gather)."""
    sk = prob.kv_lens[b]
    bs = prob.block_size
    idx = torch.arange(sk)
    pages = prob.block_table[b, (idx // bs)].long()
    slots = idx % bs
    k = prob.k_cache[pages, slots].to(torch.float64)
    v = prob.v_cache[pages, slots].to(torch.float64)
    return k, v


def torch_reference(prob):
    """Library cross-check: torch CPU float64 SDPA per sequence, K/V expanded by
    repeat_interleave for GQA, bottom-right causal mask as a boolean attn_mask."""
    outs = []
    g = prob.num_q_heads // prob.num_kv_heads
    for b in range(prob.num_seqs):
        q0, q1 = int(prob.query_start_loc[b]), int(prob.query_start_loc[b + 1])
        sq, sk = q1 - q0, prob.kv_lens[b]
        q = prob.q[q0:q1].to(torch.float64).permute(1, 0, 2)           # [H, Sq, d]
        k, v = dense_logical(prob, b)
        k = k.permute(1, 0, 2).repeat_interleave(g, dim=0)             # [H, Sk, d]
        v = v.permute(1, 0, 2).repeat_interleave(g, dim=0)
        mask = torch.ones(sq, sk, dtype=torch.bool)
        if prob.causal:
            mask = ~torch.triu(torch.ones(sq, sk, dtype=torch.bool), diagonal=sk - sq + 1)
        o = torch.nn.functional.scaled_dot_product_attention(
            q.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0), attn_mask=mask, scale=prob.scale)
        outs.append(o[0].permute(1, 0, 2).reshape(sq * prob.num_q_heads, prob.head_size))
    return torch.cat(outs).numpy()


# ----------------------------------------------------------------------------
# definition vs library
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("causal", [True, False])
def test_definition_matches_torch_sdpa(dtype, causal):
    prob = attn_inputs.paged_problem(seed=3, q_lens=[5, 17, 1, 9], kv_lens=[7, 40, 33, 9],
                                     num_q_heads=6, num_kv_heads=2, head_size=16, block_size=8,
                                     dtype=dtype, causal=causal, pool_extra=3)
    out, lse = run(prob)
    ref = torch_reference(prob)
    assert np.max(np.abs(out - ref)) < 1e-12


def test_lse_matches_logsumexp():
    prob = attn_inputs.paged_problem(seed=4, q_lens=[6], kv_lens=[11], num_q_heads=2,
                                     num_kv_heads=1, head_size=8, block_size=4, causal=True)
    _, lse = run(prob)
    k, _ = dense_logical(prob, 0)
    q = prob.q.to(torch.float64)
    for t in range(6):
        for h in range(2):
            s = prob.scale * (k[:, 0, :] @ q[t, h])
            lim = t + (11 - 6) + 1
            assert abs(lse[t * 2 + h] - torch.logsumexp(s[:lim], 0).item()) < 1e-12


# ----------------------------------------------------------------------------
# mask orientation (golden)
# ----------------------------------------------------------------------------

def _read_masks():
    cases = {}
    with open(os.path.join(GOLDEN, "causal_masks.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            left, right = line.split(":")
            sq, sk, row = (int(x) for x in left.split())
            keys = [] if right.strip() == "-" else [int(x) for x in right.split()]
            cases.setdefault((sq, sk), {})[row] = keys
    return cases


@pytest.mark.parametrize("shape", sorted(_read_masks().keys()))
def test_causal_mask_matches_golden(shape):
    """With Q = 0 every visible key gets the same weight, and with V_j the j-th
    unit vector the output row is the indicator of the visible set / its size."""
    sq, sk = shape
    golden = _read_masks()[shape]
    d = 8
    prob = attn_inputs.paged_problem(seed=0, q_lens=[sq], kv_lens=[sk], num_q_heads=1,
                                     num_kv_heads=1, head_size=d, block_size=4, causal=True,
                                     permute=False, poison=False)
    prob.q.zero_()
    for j in range(sk):
        prob.v_cache[j // 4, j % 4, 0].zero_()
        prob.v_cache[j // 4, j % 4, 0, j] = 1.0
    out, lse = run(prob)
    for i in range(sq):
        keys = golden[i]
        exp = np.zeros(d)
        if keys:
            exp[keys] = 1.0 / len(keys)
            assert abs(lse[i] - math.log(len(keys))) < 1e-12
        else:
            assert lse[i] == -math.inf
        assert np.array_equal(out[i], exp) or np.max(np.abs(out[i] - exp)) < 1e-15


# ----------------------------------------------------------------------------
# closed forms and invariants
# ----------------------------------------------------------------------------

def test_two_keys_closed_form():
    """Two visible keys: O = sigmoid(s0 - s1) V0 + sigmoid(s1 - s0) V1."""
    prob = attn_inputs.paged_problem(seed=5, q_lens=[1], kv_lens=[2], num_q_heads=1,
                                     num_kv_heads=1, head_size=4, block_size=2, causal=False,
                                     permute=False, poison=False)
    out, lse = run(prob)
    q = prob.q[0, 0].to(torch.float64).numpy()
    k = prob.k_cache[0, :, 0].to(torch.float64).numpy()
    v = prob.v_cache[0, :, 0].to(torch.float64).numpy()
    s0, s1 = prob.scale * q @ k[0], prob.scale * q @ k[1]
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    assert np.max(np.abs(out[0] - (w0 * v[0] + w1 * v[1]))) < 1e-14
    m = max(s0, s1)
    assert abs(lse[0] - (m + math.log(math.exp(s0 - m) + math.exp(s1 - m)))) < 1e-14


def test_identical_keys_give_mean_of_visible_values():
    prob = attn_inputs.paged_problem(seed=6, q_lens=[4], kv_lens=[9], num_q_heads=2,
                                     num_kv_heads=1, head_size=8, block_size=4, causal=True,
                                     poison=False, permute=False)
    key = prob.k_cache[0, 0, 0].clone()
    prob.k_cache[:, :, 0] = key
    out, _ = run(prob)
    _, v = dense_logical(prob, 0)
    for i in range(4):
        lim = i + 9 - 4 + 1
        mean = v[:lim, 0].mean(0).numpy()
        for h in range(2):
            assert np.max(np.abs(out[i * 2 + h] - mean)) < 1e-14


def test_first_causal_row_is_v0():
    prob = attn_inputs.paged_problem(seed=7, q_lens=[12], kv_lens=[12], num_q_heads=4,
                                     num_kv_heads=2, head_size=16, block_size=4, causal=True)
    out, lse = run(prob)
    _, v = dense_logical(prob, 0)
    for h in range(4):
        assert np.array_equal(out[h], v[0, h // 2].numpy())


def test_shift_invariance_of_keys():
    """Adding the same vector u to every key adds tau*<q,u> to every score of a
    row, which leaves the softmax (and O) unchanged ([ALG] sec. 2).  Keys are
    put on a grid of quarters so that K + u is exact in fp16."""
    def make():
        p = attn_inputs.paged_problem(seed=8, q_lens=[6, 3], kv_lens=[10, 7], num_q_heads=2,
                                      num_kv_heads=1, head_size=8, block_size=4, causal=True,
                                      poison=False, dtype=torch.float16)
        p.k_cache = ((p.k_cache.to(torch.float64) * 4).round() / 4).to(torch.float16)
        return p
    base = make()
    out0, _ = run(base)
    shifted = make()
    u = torch.zeros(8, dtype=torch.float64)
    u[0] = 0.5
    u[3] = -1.25
    k = shifted.k_cache.to(torch.float64) + u
    assert torch.equal(k.to(torch.float16).to(torch.float64), k)
    shifted.k_cache = k.to(torch.float16)
    out1, _ = run(shifted)
    assert np.max(np.abs(out0 - out1)) < 1e-12
    assert np.max(np.abs(out0)) > 0.1


def test_zero_query_is_prefix_mean_and_ones_give_ones():
    prob = attn_inputs.paged_problem(seed=9, q_lens=[5], kv_lens=[8], num_q_heads=1,
                                     num_kv_heads=1, head_size=4, block_size=4, causal=True,
                                     poison=False)
    prob.q.zero_()
    out, _ = run(prob)
    _, v = dense_logical(prob, 0)
    for i in range(5):
        assert np.max(np.abs(out[i] - v[:i + 4, 0].mean(0).numpy())) < 1e-14
    prob.v_cache.fill_(1.0)
    prob.q.normal_()
    prob.q.copy_(prob.q.to(torch.bfloat16))
    out, _ = run(prob)
    assert np.max(np.abs(out - 1.0)) < 1e-14


def test_convex_hull():
    prob = attn_inputs.paged_problem(seed=10, q_lens=[7, 3], kv_lens=[30, 3], num_q_heads=4,
                                     num_kv_heads=4, head_size=8, block_size=16, causal=False)
    out, _ = run(prob)
    for b in range(2):
        _, v = dense_logical(prob, b)
        q0, q1 = int(prob.query_start_loc[b]), int(prob.query_start_loc[b + 1])
        for t in range(q0, q1):
            for h in range(4):
                o = out[t * 4 + h]
                assert np.all(o <= v[:, h].max(0).values.numpy() + 1e-12)
                assert np.all(o >= v[:, h].min(0).values.numpy() - 1e-12)


def test_decode_causal_equals_noncausal():
    """A single query row attends to every key either way ([ALG] sec. 4)."""
    a = attn_inputs.paged_problem(seed=11, q_lens=[1, 1, 1], kv_lens=[5, 64, 33], num_q_heads=8,
                                  num_kv_heads=2, head_size=16, block_size=16, causal=True)
    b = attn_inputs.paged_problem(seed=11, q_lens=[1, 1, 1], kv_lens=[5, 64, 33], num_q_heads=8,
                                  num_kv_heads=2, head_size=16, block_size=16, causal=False)
    assert np.array_equal(run(a)[0], run(b)[0])


def test_gqa_equals_mha_with_repeated_kv():
    g = attn_inputs.paged_problem(seed=12, q_lens=[5, 4], kv_lens=[9, 20], num_q_heads=6,
                                  num_kv_heads=2, head_size=8, block_size=4, causal=True)
    m = attn_inputs.paged_problem(seed=12, q_lens=[5, 4], kv_lens=[9, 20], num_q_heads=6,
                                  num_kv_heads=6, head_size=8, block_size=4, causal=True)
    m.q.copy_(g.q)
    m.k_cache = g.k_cache.repeat_interleave(3, dim=2).contiguous()
    m.v_cache = g.v_cache.repeat_interleave(3, dim=2).contiguous()
    m.block_table = g.block_table.clone()
    assert np.array_equal(run(g)[0], run(m)[0])


def test_paging_is_invisible():
    """Same logical K/V under different block sizes and permutations (the
    generator draws values in logical order) gives identical results."""
    outs = []
    for bs, perm in ((4, True), (8, False), (64, True), (16, True)):
        p = attn_inputs.paged_problem(seed=13, q_lens=[7, 2], kv_lens=[19, 50], num_q_heads=2,
                                      num_kv_heads=1, head_size=8, block_size=bs, causal=True,
                                      permute=perm, pool_extra=2)
        outs.append(run(p)[0])
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)


def test_empty_rows():
    """causal with Sq > Sk leaves the first Sq - Sk rows without keys; kv_len 0
    leaves all rows without keys: output 0, lse -inf (the oracle's reading)."""
    p = attn_inputs.paged_problem(seed=14, q_lens=[6, 3], kv_lens=[2, 0], num_q_heads=1,
                                  num_kv_heads=1, head_size=4, block_size=4, causal=True)
    out, lse = run(p)
    for i in range(4):
        assert np.all(out[i] == 0) and lse[i] == -math.inf
    assert np.all(np.isfinite(out[4:6]))
    for t in range(6, 9):
        assert np.all(out[t] == 0) and lse[t] == -math.inf


def test_row_sampling_matches_full():
    p = attn_inputs.paged_problem(seed=15, q_lens=[9, 14], kv_lens=[9, 30], num_q_heads=4,
                                  num_kv_heads=2, head_size=8, block_size=8, causal=True)
    full, lse_full = run(p)
    rows = [0, 5, 37, 91, 22, 3]
    part, lse_part = run(p, rows=rows)
    assert np.array_equal(full[rows], part)
    assert np.array_equal(lse_full[rows], lse_part)


# ----------------------------------------------------------------------------
# the streaming recurrence and the split combine are exact
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("tile", [1, 3, 16, 64, 1000])
def test_streaming_recurrence_equals_definition(tile):
    p = attn_inputs.paged_problem(seed=16, q_lens=[8, 1, 20], kv_lens=[70, 129, 20],
                                  num_q_heads=4, num_kv_heads=2, head_size=16, block_size=16,
                                  causal=True, sigma=2.0)
    d_out, d_lse = run(p)
    s_out, s_lse = run(p, variant=1, param=tile)
    assert np.max(np.abs(d_out - s_out)) < 1e-12
    assert np.max(np.abs(d_lse - s_lse)) < 1e-12


@pytest.mark.parametrize("parts", [1, 2, 8, 13])
def test_split_combine_equals_definition(parts):
    p = attn_inputs.paged_problem(seed=17, q_lens=[1] * 5, kv_lens=[1, 17, 100, 512, 333],
                                  num_q_heads=8, num_kv_heads=2, head_size=16, block_size=16,
                                  causal=False, sigma=2.0)
    d_out, d_lse = run(p)
    s_out, s_lse = run(p, variant=2, param=parts)
    assert np.max(np.abs(d_out - s_out)) < 1e-12
    assert np.max(np.abs(d_lse - s_lse)) < 1e-12


# ----------------------------------------------------------------------------
# widening and rounding
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("dt,tdt", [(oracle.BF16, torch.bfloat16), (oracle.F16, torch.float16)])
def test_widen_all_patterns(dt, tdt):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.widen16(bits, dt)
    ref = torch.from_numpy(bits.view(np.int16)).view(tdt).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def _golden_rounding():
    rows = []
    with open(os.path.join(GOLDEN, "rounding_cases.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                dt, x, a, b, c = line.split()
                rows.append((dt, int(x, 16), int(a, 16), int(b, 16), int(c, 16)))
    return rows


@pytest.mark.parametrize("case", _golden_rounding())
def test_rounding_golden(case):
    dt, xbits, rtne, rtna, rtz = case
    dtype = oracle.BF16 if dt == "bf16" else oracle.F16
    x = np.array([xbits], dtype=np.uint32).view(np.float32)
    assert oracle.round_f32(x, dtype, oracle.RTNE)[0] == rtne
    assert oracle.round_f32(x, dtype, oracle.RTNA)[0] == rtna
    assert oracle.round_f32(x, dtype, oracle.RTZ)[0] == rtz


def _sample_f32(n, seed):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    return x[~np.isnan(x)]


def _brute_force(x, dtype, mode):
    """Nearest representable value by search over all finite 16-bit patterns."""
    tdt = torch.bfloat16 if dtype == oracle.BF16 else torch.float16
    pats = np.arange(0, 0x7C00 if dtype == oracle.F16 else 0x7F80, dtype=np.uint32).astype(np.uint16)
    vals = torch.from_numpy(pats.view(np.int16)).view(tdt).to(torch.float64).numpy()
    maxfin = vals[-1]
    ulp_top = vals[-1] - vals[-2]
    out = np.empty(x.shape, dtype=np.uint16)
    ax = np.abs(x.astype(np.float64))
    idx = np.searchsorted(vals, ax, side="right") - 1          # vals[idx] <= |x|
    for n in range(x.size):
        a = ax[n]
        sign = 0x8000 if np.signbit(x[n]) else 0
        if np.isinf(a):
            out[n] = sign | (0x7C00 if dtype == oracle.F16 else 0x7F80)
            continue
        i = idx[n]
        lo = vals[i]
        if lo == a:
            out[n] = sign | pats[i]
            continue
        if i + 1 < len(vals):
            hi, hi_pat = vals[i + 1], pats[i + 1]
        else:
            hi, hi_pat = maxfin + ulp_top, (0x7C00 if dtype == oracle.F16 else 0x7F80)
        if mode == oracle.RTZ:
            pick = pats[i]
        elif a - lo < hi - a:
            pick = pats[i]
        elif a - lo > hi - a:
            pick = hi_pat
        elif mode == oracle.RTNA:
            pick = hi_pat
        else:
            pick = pats[i] if pats[i] % 2 == 0 else hi_pat
        out[n] = sign | pick
    return out


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.F16])
@pytest.mark.parametrize("mode", [oracle.RTNE, oracle.RTNA, oracle.RTZ])
def test_rounding_brute_force(dtype, mode):
    x = _sample_f32(20000, seed=100 + mode)
    # add exact ties and near-ties around random representable values
    rng = np.random.default_rng(7 + mode)
    tdt = torch.bfloat16 if dtype == oracle.BF16 else torch.float16
    base = rng.integers(1, 0x7BFF if dtype == oracle.F16 else 0x7F7F, size=3000).astype(np.uint16)
    lo = torch.from_numpy(base.view(np.int16)).view(tdt).to(torch.float64).numpy()
    hi = torch.from_numpy((base + 1).view(np.int16)).view(tdt).to(torch.float64).numpy()
    mid = ((lo + hi) / 2).astype(np.float32)
    x = np.concatenate([x, mid, -mid, np.nextafter(mid, np.float32(np.inf)),
                        np.nextafter(mid, np.float32(0))]).astype(np.float32)
    ours = oracle.round_f32(x, dtype, mode)
    ref = _brute_force(x, dtype, mode)
    assert np.array_equal(ours, ref)


def test_rtne_matches_torch_cast_strided_sweep():
    bits = np.arange(0, 2**32, 4099, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    keep = ~np.isnan(x)
    x = x[keep]
    t = torch.from_numpy(x)
    for dtype, tdt in ((oracle.BF16, torch.bfloat16), (oracle.F16, torch.float16)):
        ours = oracle.round_f32(x, dtype, oracle.RTNE)
        ref = t.to(tdt).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(ours, ref)


def test_bf16_rtz_and_rtna_closed_forms():
    """bf16 shares binary32's exponent range: toward zero keeps the top 16
    bits; ties-away adds half of the dropped unit (0x8000) then keeps the top
    16 bits."""
    bits = np.arange(0, 2**32, 3001, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    keep = ~np.isnan(x)
    b = bits[keep]
    assert np.array_equal(oracle.round_f32(x[keep], oracle.BF16, oracle.RTZ),
                          (b >> 16).astype(np.uint16))
    assert np.array_equal(oracle.round_f32(x[keep], oracle.BF16, oracle.RTNA),
                          ((b.astype(np.uint64) + 0x8000) >> 16).astype(np.uint16))


def test_nan_stays_nan():
    x = np.array([np.nan, -np.nan], dtype=np.float32)
    for dt in (oracle.BF16, oracle.F16):
        for mode in (oracle.RTNE, oracle.RTNA, oracle.RTZ):
            r = oracle.widen16(oracle.round_f32(x, dt, mode), dt)
            assert np.all(np.isnan(r))


# ----------------------------------------------------------------------------
# the oracle's own threading
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("variant,param", [(0, 0), (1, 16), (2, 8)])
def test_thread_count_does_not_change_results(variant, param):
    """Rows are independent and each is computed by one thread in a fixed
    order, so the job split across threads must not change a single bit;
    every row must be written (no row left at its initial value)."""
    p = attn_inputs.paged_problem(seed=18, q_lens=[37, 1, 90], kv_lens=[50, 300, 90],
                                  num_q_heads=6, num_kv_heads=3, head_size=16, block_size=16,
                                  causal=True)
    ref_out, ref_lse = run(p, variant=variant, param=param, threads=1)
    assert np.isfinite(ref_out).all() and np.isfinite(ref_lse).all()
    for threads in (2, 3, 7, 64):
        out, lse = run(p, variant=variant, param=param, threads=threads)
        assert np.array_equal(out, ref_out) and np.array_equal(lse, ref_lse), threads

"""Randomised parity sweep: seeded random paged problems over every supported
axis -- ragged batches (including empty query ranges and zero-length KV),
every supported block size, GQA groups odd and even, head sizes 64, 128 and 256,
fp16 and bf16, causal and non-causal, all output roundings -- each compared
element by element with the fp64 oracle and, where asked, its log-sum-exp.
Sizes are kept small enough for the oracle to check every row.

Tolerance: the measured configurations draw inputs with sigma <= 1, where
|O| stays below about 2 and the absolute bound 2e-2 (fp16) / 4e-2 (bf16)
applies as it stands.  Draws with sigma = 2 give outputs up to |O| ~ 8, whose
own 16-bit rounding (up to one unit in the last place for RTZ and RTNA:
|O| * 2^-7 for bf16, |O| * 2^-10 for fp16) is a large part of that absolute
bound; for them the rounding term is added to it."""
import numpy as np
import pytest
import torch

import attn_inputs
from tests.helpers import TOL, as_rows, gpu_decode, gpu_prefill, max_err, oracle_run, to_dev, worst

pytestmark = pytest.mark.gpu

PREFILL_BLOCKS = (16, 32, 64, 128, 256)
GROUPS = ((1, 1), (2, 2), (4, 1), (4, 2), (6, 2), (8, 2), (3, 3), (16, 2), (12, 4))


ULP_REL = {torch.bfloat16: 2.0 ** -7, torch.float16: 2.0 ** -10}


def check(prob, got, ref, rounding):
    if prob.meta["sigma"] <= 1.0 or rounding == 3:
        bound = TOL[prob.dtype]
        err = max_err(got, ref)
    else:
        bound = TOL[prob.dtype]
        d = np.abs(got - ref) - np.abs(ref) * ULP_REL[prob.dtype]
        err = float(np.max(d)) if d.size else 0.0
        if np.isnan(got).any():
            err = float("inf")
    assert err <= bound, (err, worst(got, ref))


def random_prefill(seed, head_size=None):
    rng = np.random.default_rng(seed)
    hq, hkv = GROUPS[rng.integers(len(GROUPS))]
    d = int(rng.choice([64, 128]))
    d = head_size or d
    dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float16
    causal = bool(rng.random() < 0.7)
    n = int(rng.integers(1, 5))
    q_lens, kv_lens = [], []
    for _ in range(n):
        sq = int(rng.choice([0, 1, int(rng.integers(2, 300))]))
        sk = int(rng.integers(0, 600))
        if causal:
            sk = max(sk, sq) if rng.random() < 0.8 else sk   # mostly Sk >= Sq
        q_lens.append(sq)
        kv_lens.append(sk)
    if sum(q_lens) == 0:
        q_lens[0] = 5
    return attn_inputs.paged_problem(seed=seed, q_lens=q_lens, kv_lens=kv_lens, num_q_heads=hq,
                                     num_kv_heads=hkv, head_size=d,
                                     block_size=int(rng.choice(PREFILL_BLOCKS)), dtype=dtype,
                                     causal=causal, sigma=float(rng.choice([0.5, 1.0, 2.0])),
                                     pool_extra=int(rng.integers(0, 3)))


@pytest.mark.parametrize("seed", range(24))
def test_random_prefill(seed):
    check_random_prefill(random_prefill(1000 + seed), seed % 4)


@pytest.mark.parametrize("seed", range(10))
def test_random_prefill_d256(seed):
    check_random_prefill(random_prefill(3000 + seed, head_size=256), seed % 4)


def check_random_prefill(prob, rounding):
    """rounding: 0 RTNE, 1 RTNA, 2 RTZ, 3 fp32 output."""
    out, lse = gpu_prefill(prob, rounding=rounding, lse=True)
    torch.cuda.synchronize()
    ref, ref_lse = oracle_run(prob)
    got = as_rows(out)
    check(prob, got, ref, rounding)
    g = lse.cpu().numpy().reshape(-1).astype(np.float64)
    finite = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(g), finite)
    if finite.any():
        assert np.max(np.abs(g[finite] - ref_lse[finite])) < 2e-3


def random_decode(seed, head_size=None):
    rng = np.random.default_rng(seed)
    hq, hkv = GROUPS[rng.integers(len(GROUPS))]
    d = int(rng.choice([64, 128]))
    d = head_size or d
    dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float16
    n = int(rng.integers(1, 12))
    kv_lens = [int(rng.choice([0, int(rng.integers(1, 40)), int(rng.integers(40, 3000))]))
               for _ in range(n)]
    return attn_inputs.paged_problem(seed=seed, q_lens=[1] * n, kv_lens=kv_lens, num_q_heads=hq,
                                     num_kv_heads=hkv, head_size=d,
                                     block_size=int(rng.choice([16, 32, 48, 64, 128, 256])),
                                     dtype=dtype, causal=False,
                                     pool_extra=int(rng.integers(0, 5)))


@pytest.mark.parametrize("seed", range(16))
def test_random_decode(seed):
    check_random_decode(random_decode(2000 + seed), seed)


@pytest.mark.parametrize("seed", range(6))
def test_random_decode_d256(seed):
    check_random_decode(random_decode(4000 + seed, head_size=256), seed)


def check_random_decode(prob, seed):
    splits = int(np.random.default_rng(seed).choice([1, 2, 3, 8, 13]))
    out = gpu_decode(prob, splits=splits, rounding=seed % 4)
    torch.cuda.synchronize()
    ref, _ = oracle_run(prob)
    check(prob, as_rows(out), ref, seed % 4)


# ------------------------------------------------- random feature-flag draws
# Each draw picks a random subset of the flags (sliding window with random
# sides, softcap, ALiBi, sinks, fp8 E4M3 caches) on a random paged problem and
# compares output and log-sum-exp with the oracle under the same flags.

def random_flags(rng, hq):
    from tests.test_gpu_features import sink_logits, slopes
    f = {}
    if rng.random() < 0.5:
        left = int(rng.choice([-1, 0, int(rng.integers(1, 400))]))
        right = int(rng.choice([-1, 0, int(rng.integers(1, 200))]))
        if left >= 0 or right >= 0:
            f["window"] = (left, right)
    if rng.random() < 0.4:
        f["softcap"] = float(rng.choice([3.0, 15.0, 50.0]))
    if rng.random() < 0.4:
        f["alibi_slopes"] = slopes(hq) * float(rng.choice([0.05, 0.5]))
    if rng.random() < 0.4:
        f["sinks"] = sink_logits(hq, int(rng.integers(0, 1000)))
    return f


def oracle_flags(prob, flags, kv_scales):
    from oracle import oracle
    return oracle.sdpa(prob.q, prob.k_cache, prob.v_cache, prob.block_table,
                       prob.query_start_loc, prob.seq_lens, num_q_heads=prob.num_q_heads,
                       num_kv_heads=prob.num_kv_heads, head_size=prob.head_size,
                       block_size=prob.block_size, scale=prob.scale, causal=prob.causal,
                       dtype=oracle.BF16 if prob.dtype == torch.bfloat16 else oracle.F16,
                       window=flags.get("window", (-1, -1)), softcap=flags.get("softcap", 0.0),
                       alibi_slopes=None if "alibi_slopes" not in flags
                       else flags["alibi_slopes"].double().numpy(),
                       sinks=None if "sinks" not in flags else flags["sinks"].double().numpy(),
                       kv_scales=kv_scales)


def check_flagged(prob, out, lse, flags, kv_scales, rounding):
    torch.cuda.synchronize()
    ref, ref_lse = oracle_flags(prob, flags, kv_scales)
    check(prob, as_rows(out), ref, rounding)
    g = lse.cpu().numpy().reshape(-1).astype(np.float64)
    finite = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(g), finite)
    if finite.any():
        assert np.max(np.abs(g[finite] - ref_lse[finite])) < 2e-3


def on_device(flags):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in flags.items()}


@pytest.mark.parametrize("seed", range(16))
def test_random_flagged_prefill(seed):
    import attention_forward_sdpa_gb300 as attn
    rng = np.random.default_rng(5000 + seed)
    base = random_prefill(5000 + seed, head_size=int(rng.choice([64, 128, 256])))
    fp8 = rng.random() < 0.4
    prob = attn_inputs.paged_problem(seed=5000 + seed, q_lens=base.q_lens, kv_lens=base.kv_lens,
                                     num_q_heads=base.num_q_heads,
                                     num_kv_heads=base.num_kv_heads, head_size=base.head_size,
                                     block_size=base.block_size, dtype=base.dtype,
                                     causal=base.causal, sigma=min(base.meta["sigma"], 1.0),
                                     pool_extra=1, kv_dtype=torch.float8_e4m3fn if fp8 else None)
    flags = random_flags(rng, prob.num_q_heads)
    kv_scales = (prob.k_scale, prob.v_scale) if fp8 else None
    rounding = seed % 4
    t = to_dev(prob)
    out, lse = attn.prefill(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                            t["query_start_loc"], t["seq_lens"], max_seqlen_q=prob.max_seqlen_q,
                            max_seqlen_k=prob.max_seqlen_k, scale=prob.scale, causal=prob.causal,
                            rounding=rounding, return_lse=True, kv_scales=kv_scales,
                            **on_device(flags))
    check_flagged(prob, out, lse, flags, kv_scales, rounding)


@pytest.mark.parametrize("seed", range(12))
def test_random_flagged_decode(seed):
    import attention_forward_sdpa_gb300 as attn
    rng = np.random.default_rng(6000 + seed)
    base = random_decode(6000 + seed, head_size=int(rng.choice([64, 128, 256])))
    fp8 = rng.random() < 0.5
    prob = attn_inputs.paged_problem(seed=6000 + seed, q_lens=base.q_lens, kv_lens=base.kv_lens,
                                     num_q_heads=base.num_q_heads,
                                     num_kv_heads=base.num_kv_heads, head_size=base.head_size,
                                     block_size=base.block_size, dtype=base.dtype, causal=False,
                                     pool_extra=2, kv_dtype=torch.float8_e4m3fn if fp8 else None)
    flags = random_flags(rng, prob.num_q_heads)
    flags.pop("window", None)
    if rng.random() < 0.5:
        flags["window"] = (int(rng.integers(0, 1500)), -1)
    kv_scales = (prob.k_scale, prob.v_scale) if fp8 else None
    rounding = seed % 4
    splits = int(rng.choice([1, 3, 8]))
    t = to_dev(prob)
    out, lse = attn.decode(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"],
                           max_seqlen_k=prob.max_seqlen_k, scale=prob.scale, num_splits=splits,
                           rounding=rounding, return_lse=True, kv_scales=kv_scales,
                           **on_device(flags))
    check_flagged(prob, out, lse, flags, kv_scales, rounding)

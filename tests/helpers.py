"""Shared helpers for the GPU parity tests: move a seeded problem to the device,
run the library through its binding, run the oracle, compare."""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle

TOL = {torch.bfloat16: 4e-2, torch.float16: 2e-2}   # max |err| vs the fp64 oracle
FIELDS = ("q", "k_cache", "v_cache", "block_table", "query_start_loc", "seq_lens")


def to_dev(prob, dev="cuda"):
    return {k: getattr(prob, k).to(dev) for k in FIELDS}


def gpu_prefill(prob, t=None, rounding=0, lse=False, status=None):
    import attention_forward_sdpa_gb300 as attn
    t = t or to_dev(prob)
    return attn.prefill(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                        t["query_start_loc"], t["seq_lens"], max_seqlen_q=prob.max_seqlen_q,
                        max_seqlen_k=prob.max_seqlen_k, scale=prob.scale, causal=prob.causal,
                        rounding=rounding, return_lse=lse, status=status)


def gpu_decode(prob, t=None, splits=8, rounding=0, lse=False, status=None, workspace=None,
               **features):
    import attention_forward_sdpa_gb300 as attn
    t = t or to_dev(prob)
    return attn.decode(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"],
                       max_seqlen_k=prob.max_seqlen_k, scale=prob.scale, num_splits=splits,
                       rounding=rounding, return_lse=lse, status=status, workspace=workspace,
                       **features)


def oracle_run(prob, rows=None, threads=None):
    return oracle.sdpa(prob.q, prob.k_cache, prob.v_cache, prob.block_table,
                       prob.query_start_loc, prob.seq_lens, num_q_heads=prob.num_q_heads,
                       num_kv_heads=prob.num_kv_heads, head_size=prob.head_size,
                       block_size=prob.block_size, scale=prob.scale, causal=prob.causal,
                       dtype=oracle.BF16 if prob.dtype == torch.bfloat16 else oracle.F16,
                       rows=rows, n_threads=threads)


def as_rows(out: torch.Tensor) -> np.ndarray:
    """[tokens, heads, d] device tensor -> float64 [tokens*heads, d] host array."""
    return out.float().cpu().numpy().reshape(-1, out.shape[-1]).astype(np.float64)


def max_err(got_rows: np.ndarray, ref: np.ndarray) -> float:
    if got_rows.size == 0:
        return 0.0
    d = np.abs(got_rows - ref)
    if np.isnan(d).any():
        return float("inf")
    return float(d.max())


def sample_rows(prob, per_head_random=64, seed=1):
    """Every (sequence, head): rows 0, 1, last-1, last, plus random rows."""
    rng = np.random.default_rng(seed)
    rows = []
    H = prob.num_q_heads
    for b in range(prob.num_seqs):
        q0, q1 = int(prob.query_start_loc[b]), int(prob.query_start_loc[b + 1])
        n = q1 - q0
        if n == 0:
            continue
        fixed = sorted({0, min(1, n - 1), max(0, n - 2), n - 1})
        rand = rng.integers(0, n, size=min(per_head_random, n)).tolist()
        for h in range(H):
            for i in fixed + rand:
                rows.append((q0 + i) * H + h)
    return np.array(sorted(set(rows)), dtype=np.int64)


def worst(got_rows, ref, n=5):
    d = np.abs(got_rows - ref)
    flat = np.argsort(d, axis=None)[::-1][:n]
    return [(int(i // d.shape[1]), int(i % d.shape[1]), float(got_rows.flat[i]), float(ref.flat[i]))
            for i in flat]


# ----------------------------------------------------------------------------
# parity report: per checked case, max |err|, mean |err| and the largest error
# in units of the output format's spacing at the reference value (ULP)
# ----------------------------------------------------------------------------

PARITY = []
_MANT = {torch.bfloat16: 7, torch.float16: 10}
_MIN_EXP = {torch.bfloat16: -126, torch.float16: -14}


def ulp_of(ref: np.ndarray, dtype) -> np.ndarray:
    """Spacing of the 16-bit format at |ref| (its subnormal spacing below the
    smallest normal)."""
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, _MIN_EXP[dtype])
    return np.exp2(e - _MANT[dtype])


ULP_FLOOR = 2.0 ** -6   # below this |ref| the absolute error is the meaningful one


def record(name: str, got: np.ndarray, ref: np.ndarray, dtype) -> dict:
    """ULP counts are taken where |ref| >= ULP_FLOOR (near zero the format's
    spacing is far finer than the fp32 accumulation error, and the absolute
    error is reported instead); p99.9 is over those elements."""
    d = np.abs(got - ref)
    fin = np.isfinite(ref)
    big = fin & (np.abs(ref) >= ULP_FLOOR)
    u = d[big] / ulp_of(ref[big], dtype) if big.any() else np.zeros(1)
    row = {"case": name, "elements": int(got.size),
           "max_abs": float(d[fin].max()) if fin.any() else 0.0,
           "mean_abs": float(d[fin].mean()) if fin.any() else 0.0,
           "max_ulp": float(u.max()), "p999_ulp": float(np.percentile(u, 99.9))}
    PARITY.append(row)
    return row

"""GPU parity of the feature-flagged variants (sliding window, softcap, ALiBi,
sinks; named in "gfx942 unified attention, from the math up", sec. 9) against
the fp64 oracle, for the paged prefill (head sizes 64, 128, 256; GQA pairs of
heads and row-block pairs), the dense strided entry point, and decode (the
tcgen05 split kernel at head size 128, the SIMT one otherwise, plus the merge;
one and several splits).

Tolerance: 2e-2 (fp16) / 4e-2 (bf16) max |err|, as for the plain calls.  The
windows are chosen so that whole key tiles fall left of every row of a query
tile (the kernels skip those tiles) and so that the per-element masks cut
through tiles on both sides.  The log-sum-exp includes the sink.
"""
import numpy as np
import pytest
import torch

import attn_inputs
from oracle import oracle
from tests.helpers import TOL, as_rows, gpu_decode, gpu_prefill, max_err, to_dev, worst

pytestmark = pytest.mark.gpu


def slopes(h):
    return torch.tensor([2.0 ** (-8.0 * (i + 1) / h) for i in range(h)], dtype=torch.float32)


def sink_logits(h, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(h, generator=g, dtype=torch.float32) * 2.0


def oracle_feat(prob, window=None, softcap=0.0, alibi_slopes=None, sinks=None):
    return oracle.sdpa(prob.q, prob.k_cache, prob.v_cache, prob.block_table,
                       prob.query_start_loc, prob.seq_lens, num_q_heads=prob.num_q_heads,
                       num_kv_heads=prob.num_kv_heads, head_size=prob.head_size,
                       block_size=prob.block_size, scale=prob.scale, causal=prob.causal,
                       dtype=oracle.BF16 if prob.dtype == torch.bfloat16 else oracle.F16,
                       window=window if window is not None else (-1, -1), softcap=softcap,
                       alibi_slopes=None if alibi_slopes is None else alibi_slopes.double().numpy(),
                       sinks=None if sinks is None else sinks.double().numpy())


def on_gpu(feat):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in feat.items()}


def features(kind, h, seed):
    if kind == "window_causal":
        return dict(window=(200, -1))
    if kind == "window_band":
        return dict(window=(150, 90))
    if kind == "softcap":
        return dict(softcap=4.0)
    if kind == "softcap_wide":
        return dict(softcap=30.0)
    if kind == "alibi":
        return dict(alibi_slopes=slopes(h))
    if kind == "sinks":
        return dict(sinks=sink_logits(h, seed))
    if kind == "all":
        return dict(window=(260, 40), softcap=6.0, alibi_slopes=slopes(h) * 0.1,
                    sinks=sink_logits(h, seed))
    raise KeyError(kind)


KINDS = ("window_causal", "window_band", "softcap", "softcap_wide", "alibi", "sinks", "all")
SHAPES = {
    # d, Hq, Hkv, dtype, block size
    "d128_gqa4_bf16": (128, 8, 2, torch.bfloat16, 64),
    "d64_gqa3_fp16": (64, 6, 2, torch.float16, 32),      # odd group: row-block pairs
    "d256_gqa2_bf16": (256, 4, 2, torch.bfloat16, 16),
}


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("kind", KINDS)
def test_prefill_features(shape, kind):
    d, hq, hkv, dtype, bs = SHAPES[shape]
    causal = kind != "window_band"
    prob = attn_inputs.paged_problem(seed=81, q_lens=[700, 1, 130], kv_lens=[900, 300, 130],
                                     num_q_heads=hq, num_kv_heads=hkv, head_size=d, block_size=bs,
                                     dtype=dtype, causal=causal, sigma=1.5, pool_extra=3)
    feat = features(kind, hq, 5)
    out, lse = gpu_prefill_feat(prob, on_gpu(feat))
    torch.cuda.synchronize()
    ref, ref_lse = oracle_feat(prob, **feat)
    got = as_rows(out)
    err = max_err(got, ref)
    assert err <= TOL[dtype], (err, worst(got, ref))
    g = lse.cpu().numpy().reshape(-1).astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(g), fin)
    assert np.max(np.abs(g[fin] - ref_lse[fin])) < 2e-3


def gpu_prefill_feat(prob, feat, rounding=0):
    import attention_forward_sdpa_gb300 as attn
    t = to_dev(prob)
    return attn.prefill(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                        t["query_start_loc"], t["seq_lens"], max_seqlen_q=prob.max_seqlen_q,
                        max_seqlen_k=prob.max_seqlen_k, scale=prob.scale, causal=prob.causal,
                        rounding=rounding, return_lse=True, **feat)


def test_window_skips_tiles_and_rows_without_keys_report_the_sink():
    """A short window over a long sequence (most key tiles skipped), queries
    longer than keys (rows with no visible key), sinks: O = 0 and lse = z there."""
    prob = attn_inputs.paged_problem(seed=82, q_lens=[300, 2000], kv_lens=[100, 2000],
                                     num_q_heads=4, num_kv_heads=2, head_size=128, block_size=64,
                                     causal=True)
    feat = dict(window=(64, -1), sinks=sink_logits(4, 6))
    out, lse = gpu_prefill_feat(prob, on_gpu(feat))
    torch.cuda.synchronize()
    ref, ref_lse = oracle_feat(prob, **feat)
    got = as_rows(out)
    assert max_err(got, ref) <= TOL[prob.dtype]
    g = lse.cpu().numpy().reshape(-1).astype(np.float64)
    empty = np.all(ref == 0, axis=1)
    assert empty.sum() > 0 and np.all(got[empty] == 0)
    assert np.max(np.abs(g - ref_lse)) < 2e-3


def test_plain_flags_equal_the_plain_call_bitwise():
    """Flags that change nothing (an unbounded window, zero slopes, sinks at
    -inf) take the feature kernels and must reproduce the plain kernels bit
    for bit (same arithmetic on the same tiles)."""
    prob = attn_inputs.paged_problem(seed=83, q_lens=[300, 77], kv_lens=[520, 77], num_q_heads=4,
                                     num_kv_heads=2, head_size=128, block_size=64, causal=True)
    plain = gpu_prefill(prob)
    feat = dict(window=(100000, 100000), sinks=torch.full((4,), -float("inf")))
    out, _ = gpu_prefill_feat(prob, on_gpu(feat))
    torch.cuda.synchronize()
    assert torch.equal(plain, out)


@pytest.mark.parametrize("rounding", [1, 2, 3])
def test_features_with_other_roundings(rounding):
    prob = attn_inputs.paged_problem(seed=84, q_lens=[260], kv_lens=[400], num_q_heads=4,
                                     num_kv_heads=4, head_size=128, block_size=128, causal=False)
    feat = features("all", 4, 7)
    out, _ = gpu_prefill_feat(prob, on_gpu(feat), rounding=rounding)
    torch.cuda.synchronize()
    ref, _ = oracle_feat(prob, **feat)
    assert max_err(as_rows(out), ref) <= TOL[prob.dtype]


@pytest.mark.parametrize("layout", ["bshd", "bhsd"])
def test_dense_features_equal_paged(layout):
    from tests.test_gpu_dense import make, run_dense
    import attention_forward_sdpa_gb300 as attn
    B, Sq, Sk, Hq, Hkv = 2, 256, 384, 8, 2
    prob = make(B, Sq, Sk, Hq, Hkv, 128, torch.bfloat16, True, seed=85)
    feat = on_gpu(features("all", Hq, 8))
    from tests.test_gpu_dense import dense_tensors
    q, k, v = dense_tensors(prob, B, Sq, Sk, layout)
    res = attn.dense(q, k, v, layout=layout, scale=prob.scale, causal=True, **feat)
    out = (res if layout == "bshd" else res.transpose(1, 2)).contiguous().view(B * Sq, Hq, 128)
    paged, _ = gpu_prefill_feat(prob, feat)
    torch.cuda.synchronize()
    assert torch.equal(out, paged)
    ref, _ = oracle_feat(prob, **features("all", Hq, 8))
    assert max_err(as_rows(out), ref) <= TOL[torch.bfloat16]


# ---------------------------------------------------------------- decode

@pytest.mark.parametrize("splits", [1, 8])
@pytest.mark.parametrize("kind", ("window_causal", "softcap", "alibi", "sinks", "all"))
@pytest.mark.parametrize("d,hq,hkv", [(128, 32, 8), (128, 16, 2), (64, 6, 2), (64, 16, 4),
                                      (256, 8, 2)])
def test_decode_features(splits, kind, d, hq, hkv):
    prob = attn_inputs.paged_problem(seed=86, q_lens=[1] * 6, kv_lens=[1, 17, 0, 300, 2049, 700],
                                     num_q_heads=hq, num_kv_heads=hkv, head_size=d, block_size=16,
                                     causal=False, sigma=1.5, pool_extra=4)
    feat = features(kind, hq, 9)
    if kind == "window_causal":
        feat = dict(window=(200, -1))
    out, lse = gpu_decode(prob, splits=splits, lse=True, **on_gpu(feat))
    torch.cuda.synchronize()
    ref, ref_lse = oracle_feat(prob, **feat)
    got = as_rows(out)
    err = max_err(got, ref)
    assert err <= TOL[prob.dtype], (err, worst(got, ref))
    g = lse.cpu().numpy().reshape(-1).astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(g), fin)
    assert np.max(np.abs(g[fin] - ref_lse[fin])) < 2e-3


def test_graph_wrapper_runs_flagged_decode_eagerly():
    import attention_forward_sdpa_gb300 as attn
    from attention_forward_sdpa_gb300 import graphs
    prob = attn_inputs.paged_problem(seed=87, q_lens=[1] * 4, kv_lens=[5, 64, 1000, 333],
                                     num_q_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                                     causal=False)
    t = to_dev(prob)
    out = torch.empty_like(t["q"])
    ws = torch.empty(attn.attn_decode_workspace_size(4, 8, 128, 8), dtype=torch.uint8,
                     device="cuda")
    cache = graphs.GraphCache()
    feat = dict(softcap=3.0)
    used = graphs.decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                         t["seq_lens"], max_seqlen_k=prob.max_seqlen_k, scale=prob.scale,
                         num_splits=8, workspace=ws, cache=cache, **feat)
    torch.cuda.synchronize()
    assert used is False and len(cache) == 0
    ref, _ = oracle_feat(prob, **feat)
    assert max_err(as_rows(out), ref) <= TOL[prob.dtype]

"""CUDA-graph replay through attention_forward_sdpa_gb300.graphs (the graph
heuristic of "gfx942 unified attention, from the math up" sec. 9: decode and
short prefill are replayed, long prefill runs eagerly): the replayed result
matches the fp64 oracle within the parity tolerance (4e-2 bf16), equals the
eager call bit for bit, reads the tensors' current values at replay time,
and long prefill stays eager."""
import dataclasses

import pytest
import torch

import attn_inputs
from tests.helpers import (TOL, as_rows, gpu_decode, gpu_prefill, max_err, oracle_run, to_dev,
                           worst)

pytestmark = pytest.mark.gpu


def _against_oracle(out, prob):
    torch.cuda.synchronize()
    got = as_rows(out)
    ref, _ = oracle_run(prob)
    err = max_err(got, ref)
    assert err <= TOL[prob.dtype], (err, worst(got, ref))


def test_graphed_decode_matches_eager_and_follows_new_values():
    import attention_forward_sdpa_gb300 as attn
    from attention_forward_sdpa_gb300 import graphs
    prob = attn_inputs.paged_problem(seed=21, q_lens=[1] * 5, kv_lens=[70, 900, 33, 1500, 400],
                                     num_q_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                                     dtype=torch.bfloat16, causal=False)
    t = to_dev(prob)
    cache = graphs.GraphCache()
    ws = torch.empty(attn.attn_decode_workspace_size(5, 8, 128, 8), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(t["q"])
    args = (out, t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"])
    kw = dict(max_seqlen_k=prob.max_seqlen_k, scale=prob.scale, num_splits=8, workspace=ws,
              cache=cache)
    graphs.decode(*args, **kw)                 # captured (and run once eagerly)
    graphs.decode(*args, **kw)                 # replayed
    torch.cuda.synchronize()
    assert cache.captures == 1 and cache.replays == 1
    _against_oracle(out, prob)
    assert torch.equal(out, gpu_decode(prob, t=t))
    # new values in the same tensors: the replay reads them
    t["q"].mul_(-1.0)
    graphs.decode(*args, **kw)
    torch.cuda.synchronize()
    assert cache.replays == 2
    _against_oracle(out, dataclasses.replace(prob, q=prob.q.neg()))
    assert torch.equal(out, gpu_decode(prob, t=t))


def test_graphed_short_prefill_and_eager_long_prefill():
    from attention_forward_sdpa_gb300 import graphs
    cache = graphs.GraphCache()
    short = attn_inputs.paged_problem(seed=22, q_lens=[200, 33], kv_lens=[200, 300],
                                      num_q_heads=8, num_kv_heads=2, head_size=128, block_size=64,
                                      dtype=torch.bfloat16, causal=True)
    t = to_dev(short)
    out = torch.empty_like(t["q"])
    kw = dict(max_seqlen_q=short.max_seqlen_q, max_seqlen_k=short.max_seqlen_k, scale=short.scale,
              causal=True, cache=cache)
    for _ in range(3):
        assert graphs.prefill(out, t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                              t["query_start_loc"], t["seq_lens"], **kw)
    torch.cuda.synchronize()
    assert cache.captures == 1 and cache.replays == 2
    _against_oracle(out, short)
    assert torch.equal(out, gpu_prefill(short, t=t))
    long = attn_inputs.paged_problem(seed=23, q_lens=[1024], kv_lens=[1024], num_q_heads=4,
                                     num_kv_heads=2, head_size=128, block_size=64,
                                     dtype=torch.bfloat16, causal=True)
    tl = to_dev(long)
    outl = torch.empty_like(tl["q"])
    assert not graphs.prefill(outl, tl["q"], tl["k_cache"], tl["v_cache"], tl["block_table"],
                              tl["query_start_loc"], tl["seq_lens"], max_seqlen_q=1024,
                              max_seqlen_k=1024, scale=long.scale, causal=True, cache=cache)
    torch.cuda.synchronize()
    assert len(cache) == 1                     # the long prefill was not captured
    _against_oracle(outl, long)
    assert torch.equal(outl, gpu_prefill(long, t=tl))

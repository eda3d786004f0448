"""GPU checks of the library's tensor-map cache: a repeated call on the same
buffers encodes no TMA descriptor again and gives the same bits; a call on a
new buffer of the same shape encodes that buffer's descriptor and is still
right (the cache key holds the address)."""
import numpy as np
import pytest
import torch

import attn_inputs
from tests.helpers import TOL, as_rows, max_err, oracle_run, to_dev

pytestmark = pytest.mark.gpu


def call(attn, prob, t, out):
    attn.attn_fwd_prefill(out, t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                          t["query_start_loc"], t["seq_lens"], max_seqlen_q=prob.max_seqlen_q,
                          max_seqlen_k=prob.max_seqlen_k, scale=prob.scale, causal=True)


def test_repeated_prefill_hits_the_cache():
    import attention_forward_sdpa_gb300 as attn
    prob = attn_inputs.paged_problem(seed=71, q_lens=[300, 77], kv_lens=[300, 200],
                                     num_q_heads=8, num_kv_heads=2, head_size=128, block_size=64)
    t = to_dev(prob)
    out = torch.empty_like(t["q"])
    call(attn, prob, t, out)
    torch.cuda.synchronize()
    first = out.clone()
    h0, m0 = attn.attn_tensor_map_cache_stats()
    call(attn, prob, t, out)
    torch.cuda.synchronize()
    h1, m1 = attn.attn_tensor_map_cache_stats()
    assert m1 == m0                      # nothing encoded again
    assert h1 - h0 >= 4                  # Q, K, V, O served from the cache
    assert torch.equal(first.view(torch.int16), out.view(torch.int16))
    # a new output buffer of the same shape: its map is encoded, the rest hit
    out2 = torch.empty_like(out)
    call(attn, prob, t, out2)
    torch.cuda.synchronize()
    h2, m2 = attn.attn_tensor_map_cache_stats()
    assert m2 - m1 == 1 and h2 - h1 >= 3
    assert torch.equal(first.view(torch.int16), out2.view(torch.int16))
    ref, _ = oracle_run(prob)
    assert max_err(as_rows(out2), ref) <= TOL[prob.dtype]


def test_repeated_decode_hits_the_cache():
    import attention_forward_sdpa_gb300 as attn
    prob = attn_inputs.paged_problem(seed=72, q_lens=[1] * 5, kv_lens=[700, 33, 1500, 0, 64],
                                     num_q_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                                     causal=False)
    t = to_dev(prob)
    out = torch.empty_like(t["q"])
    ws = torch.empty(attn.attn_decode_workspace_size(5, 8, 128, 8), dtype=torch.uint8,
                     device="cuda")
    outs = []
    for _ in range(3):
        attn.attn_fwd_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                             t["seq_lens"], max_seqlen_k=prob.max_seqlen_k, scale=prob.scale,
                             num_splits=8, workspace=ws)
        torch.cuda.synchronize()
        outs.append((out.clone(), attn.attn_tensor_map_cache_stats()))
    (o0, s0), (o1, s1), (o2, s2) = outs
    assert s2[1] == s1[1]                # the third call encodes nothing
    assert torch.equal(o0.view(torch.int16), o2.view(torch.int16))
    ref, _ = oracle_run(prob)
    assert max_err(as_rows(o2), ref) <= TOL[prob.dtype]

"""attn_fwd_decode_noalloc: the decode entry point for callers that may not
allocate device memory (a latency-critical serving loop that cannot afford
cudaMalloc, or a host framework / plugin interface that only hands the
library input and output pointers).  It keeps the split partials in a
library-owned device array instead of a caller workspace.

Checked through the C ABI against attn_fwd_decode (the same kernels with a
torch-allocated workspace), within the decode tests' tolerance, on two calls
in a row with different problems -- the second call reuses the array that
the first one left behind.  This file is collected last so that a run that
stops at the first failure has already run every other test; it also passes
on its own in a fresh process.
"""
import pytest
import torch

import attention_forward_sdpa_gb300 as attn
import attn_inputs
from tests.helpers import TOL, to_dev

pytestmark = pytest.mark.gpu


def _both(prob, splits):
    t = to_dev(prob)
    ref = attn.decode(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"],
                      max_seqlen_k=prob.max_seqlen_k, scale=prob.scale, num_splits=splits)
    out = torch.empty_like(t["q"])
    attn.attn_fwd_decode_noalloc(out, t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                 t["seq_lens"], max_seqlen_k=prob.max_seqlen_k, scale=prob.scale,
                                 num_splits=splits)
    torch.cuda.synchronize()
    return ref, out


def test_noalloc_matches_workspace_entry_two_calls_in_a_row():
    first = attn_inputs.paged_problem(seed=91, q_lens=[1] * 24,
                                      kv_lens=[17 + 331 * i for i in range(24)], num_q_heads=32,
                                      num_kv_heads=8, head_size=128, block_size=16, causal=False)
    second = attn_inputs.paged_problem(seed=92, q_lens=[1] * 5, kv_lens=[9, 4000, 1, 640, 2222],
                                       num_q_heads=8, num_kv_heads=2, head_size=128,
                                       block_size=32, causal=False)
    for prob, splits in ((first, 8), (second, 5)):
        ref, out = _both(prob, splits)
        diff = (ref.float() - out.float()).abs().max().item()
        assert diff <= TOL[prob.dtype], diff
        assert torch.equal(ref, out)


def test_noalloc_rejects_problems_beyond_its_scratch():
    limit = 16 * 1024 * 1024
    need = attn.attn_decode_workspace_size(4096, 32, 128, 64)
    assert need > limit
    q = torch.zeros(4096, 32, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 16, 8, 128, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(4096, 1, dtype=torch.int32, device="cuda")
    sl = torch.ones(4096, dtype=torch.int32, device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd_decode_noalloc(torch.empty_like(q), q, k, k, bt, sl, max_seqlen_k=16,
                                     scale=0.088, num_splits=64)
    assert e.value.status == 4

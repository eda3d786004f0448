"""The Python binding's own checks on CUDA tensors: arrays the kernels write
(lse, status) must have the sizes the call implies, and tensors of the wrong
rank are refused with a message, before anything reaches the library."""
import pytest
import torch

import attn_inputs
from tests.helpers import to_dev

pytestmark = pytest.mark.gpu


def small_problem():
    return attn_inputs.paged_problem(seed=5, q_lens=[3, 70], kv_lens=[40, 70], num_q_heads=4,
                                     num_kv_heads=2, head_size=128, block_size=16,
                                     dtype=torch.bfloat16, causal=True)


def prefill_call(t, prob, **kw):
    import attention_forward_sdpa_gb300 as attn
    out = torch.empty_like(t["q"])
    attn.attn_fwd_prefill(out, t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                          t["query_start_loc"], t["seq_lens"], max_seqlen_q=prob.max_seqlen_q,
                          max_seqlen_k=prob.max_seqlen_k, scale=prob.scale, causal=True, **kw)
    return out


def test_lse_of_the_wrong_shape_is_refused():
    prob = small_problem()
    t = to_dev(prob)
    total_q, hq = t["q"].shape[:2]
    with pytest.raises(ValueError, match="lse"):
        prefill_call(t, prob, lse=torch.empty(total_q * hq - 1, dtype=torch.float32, device="cuda"))
    with pytest.raises(ValueError, match="lse"):
        prefill_call(t, prob, lse=torch.empty(hq, total_q, dtype=torch.float32, device="cuda"))
    lse = torch.empty(total_q, hq, dtype=torch.float32, device="cuda")
    prefill_call(t, prob, lse=lse)
    torch.cuda.synchronize()
    assert torch.isfinite(lse).all()


def test_empty_status_word_is_refused():
    prob = small_problem()
    t = to_dev(prob)
    with pytest.raises(ValueError, match="status"):
        prefill_call(t, prob, status=torch.empty(0, dtype=torch.int32, device="cuda"))


def test_wrong_rank_is_refused():
    prob = small_problem()
    t = to_dev(prob)
    t["q"] = t["q"].reshape(t["q"].shape[0], -1)
    with pytest.raises(ValueError, match="q must be 3-D"):
        prefill_call(t, prob)


def test_decode_lse_shape_is_checked():
    import attention_forward_sdpa_gb300 as attn
    prob = attn_inputs.paged_problem(seed=6, q_lens=[1, 1], kv_lens=[40, 300], num_q_heads=8,
                                     num_kv_heads=2, head_size=128, block_size=16,
                                     dtype=torch.bfloat16, causal=False)
    t = to_dev(prob)
    out = torch.empty_like(t["q"])
    n = attn.attn_decode_workspace_size(2, 8, 128, 8)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError, match="lse"):
        attn.attn_fwd_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                             t["seq_lens"], max_seqlen_k=prob.max_seqlen_k, scale=prob.scale,
                             num_splits=8, workspace=ws,
                             lse=torch.empty(8, 2, dtype=torch.float32, device="cuda"))

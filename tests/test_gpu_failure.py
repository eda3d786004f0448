"""Failure detection on the GPU without a fault: every pipeline wait of the
prefill kernel is bounded; when one runs out the CTA raises its abort flag,
releases its tensor memory and records ATTN_ERR_TIMEOUT in the caller's
status word, and the device stays usable.  The test hook makes the first wait
run out (its producer issues no copy, so no barrier is ever completed) with a
20 ms limit, then checks the status, that the output was not touched, and that
a normal call right after it is correct.  Nothing traps, faults or hangs.
"""
import ctypes
import time

import pytest
import torch

import attn_inputs
from tests.helpers import TOL, as_rows, gpu_prefill, max_err, oracle_run, to_dev

pytestmark = pytest.mark.gpu

ATTN_ERR_TIMEOUT = 6


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


# Head size 256 runs its own kernel (one query tile per CTA, two score
# buffers); its waits are bounded the same way.
@pytest.mark.parametrize("head_size", [128, 256])
@pytest.mark.parametrize("seqs", [2, 40])
def test_prefill_wait_timeout_is_reported_and_device_stays_usable(seqs, head_size):
    import attention_forward_sdpa_gb300 as attn
    lib = attn.load_library()
    prob = attn_inputs.paged_problem(seed=11, q_lens=[150] * seqs, kv_lens=[300] * seqs,
                                     num_q_heads=8, num_kv_heads=2, head_size=head_size, block_size=64,
                                     dtype=torch.bfloat16, causal=True)
    t = to_dev(prob)
    out = torch.zeros_like(t["q"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    t0 = time.time()
    rc = lib.attn_test_prefill_timeout(
        _ptr(out), _ptr(t["q"]), _ptr(t["k_cache"]), _ptr(t["v_cache"]), _ptr(t["block_table"]),
        t["block_table"].shape[1], _ptr(t["query_start_loc"]), _ptr(t["seq_lens"]), prob.num_seqs,
        prob.max_seqlen_q, prob.max_seqlen_k, prob.total_q, 8, 2, head_size, 64,
        prob.k_cache.shape[0], prob.scale, 1, attn.BF16, 0, _ptr(status), 20_000_000,
        ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert status.item() == ATTN_ERR_TIMEOUT
    assert elapsed < 3.0, elapsed                      # bounded by the 20 ms limit, not the 4 s default
    assert torch.count_nonzero(out).item() == 0        # nothing written
    # the context is intact: the next ordinary call succeeds and is correct
    status.zero_()
    good = gpu_prefill(prob, t=t, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    ref, _ = oracle_run(prob)
    assert max_err(as_rows(good), ref) <= TOL[torch.bfloat16]

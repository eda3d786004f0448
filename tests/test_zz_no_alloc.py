"""attn_fwd_decode_noalloc: the decode entry point for callers that may not
allocate device memory (a latency-critical serving loop that cannot afford
cudaMalloc, or a host framework / plugin interface that only hands the
library input and output pointers).  It keeps the split partials in a
library-owned device array instead of a caller workspace.

Checked through the C ABI against the fp64 oracle (the decode tests'
tolerance, 4e-2 for bf16) and against attn_fwd_decode (the same kernels with
a torch-allocated workspace, bit for bit), on calls in a row with different
problems -- each call reuses the array that the one before left behind: the
tcgen05 kernel's shapes with several splits and with one, the SIMT kernel's
shapes (query-head group of 3), and the largest problem whose partials fit
the array.  The smallest problem that does not fit is refused before any
launch.  This file is collected last so that a run that stops at the first
failure has already run every other test; it also passes on its own in a
fresh process.
"""
import pytest
import torch

import attention_forward_sdpa_gb300 as attn
import attn_inputs
from tests.helpers import TOL, as_rows, max_err, oracle_run, to_dev, worst

pytestmark = pytest.mark.gpu

LIMIT = 16 * 1024 * 1024          # ATTN_DECODE_NOALLOC_SCRATCH_BYTES


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


def _check(prob, splits):
    ref, out = _both(prob, splits)
    got = as_rows(out)
    want, _ = oracle_run(prob)
    err = max_err(got, want)
    assert err <= TOL[prob.dtype], (err, worst(got, want))
    assert torch.equal(ref, out)


def _decode_problem(seed, kv_lens, hq, hkv, d, bs=16):
    return attn_inputs.paged_problem(seed=seed, q_lens=[1] * len(kv_lens), kv_lens=kv_lens,
                                     num_q_heads=hq, num_kv_heads=hkv, head_size=d,
                                     block_size=bs, causal=False)


def test_noalloc_matches_oracle_and_workspace_entry_calls_in_a_row():
    cases = [
        # tcgen05 kernel, GQA 4:1, several splits
        (_decode_problem(91, [17 + 331 * i for i in range(24)], 32, 8, 128), 8),
        # tcgen05 kernel, another block size and split count
        (_decode_problem(92, [9, 4000, 1, 640, 2222], 8, 2, 128, bs=32), 5),
        # one split: the kernel writes the output itself, the array holds the counter only
        (_decode_problem(93, [300, 1, 2500, 77], 16, 2, 128), 1),
        # SIMT kernel (query-head group of 3), head size 64
        (_decode_problem(94, [513, 2, 1200, 64, 999], 6, 2, 64), 4),
        # SIMT kernel at head size 128, after the others
        (_decode_problem(95, [1000, 31, 260], 12, 4, 128), 3),
    ]
    for prob, splits in cases:
        _check(prob, splits)


def test_noalloc_largest_problem_that_fits_and_smallest_that_does_not():
    # partials of R = seqs * heads * splits rows need R * (128 + 2) * 4 + 256
    # bytes: R = 32263 (4609 sequences, 7 splits) is the largest R that fits
    # 16 MiB, R = 32264 (4033 sequences, 8 splits) the smallest that does not
    fits = attn.attn_decode_workspace_size(4609, 1, 128, 7)
    over = attn.attn_decode_workspace_size(4033, 1, 128, 8)
    assert fits <= LIMIT < over and over - fits == 520
    g = torch.Generator().manual_seed(5)
    kv = torch.randint(1, 40, (4609,), generator=g).tolist()
    prob = _decode_problem(96, kv, 1, 1, 128)
    _check(prob, 7)
    q = torch.zeros(4033, 1, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 16, 1, 128, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(4033, 1, dtype=torch.int32, device="cuda")
    sl = torch.ones(4033, dtype=torch.int32, device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd_decode_noalloc(torch.empty_like(q), q, k, k, bt, sl, max_seqlen_k=16,
                                     scale=0.088, num_splits=8)
    assert e.value.status == 4          # ATTN_ERR_WORKSPACE
    # a much larger problem is refused the same way
    need = attn.attn_decode_workspace_size(4096, 32, 128, 64)
    assert need > LIMIT
    q = torch.zeros(4096, 32, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 16, 8, 128, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(4096, 1, dtype=torch.int32, device="cuda")
    sl = torch.ones(4096, dtype=torch.int32, device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd_decode_noalloc(torch.empty_like(q), q, k, k, bt, sl, max_seqlen_k=16,
                                     scale=0.088, num_splits=64)
    assert e.value.status == 4

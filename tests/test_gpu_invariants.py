"""GPU invariants that hold exactly or within one unit in the last place,
independent of the oracle ("gfx942 unified attention, from the math up":
sec. 1 defines O as a convex combination of V rows, sec. 4 aligns the causal
mask bottom-right, sec. 8 makes the split of the keys irrelevant):
  - V = 1 everywhere gives O = 1 within one ULP of the output format (P is
    rounded to 16 bits before P.V while the denominator keeps fp32 p, so O is
    1 up to that rounding);
  - with Sq = Sk the first causal row sees only key 0: P = 1 exactly and O is
    V_0 bit for bit, in every rounding mode;
  - decode with one split and with eight agree within the tolerance;
  - every output lies within [min V, max V] of its head's visible rows, up
    to one ULP."""
import numpy as np
import pytest
import torch

import attn_inputs
from tests.helpers import TOL, gpu_decode, gpu_prefill, to_dev, ulp_of

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_unit_values_give_unit_output(dtype, d):
    prob = attn_inputs.paged_problem(seed=41, q_lens=[300, 7], kv_lens=[300, 900], num_q_heads=4,
                                     num_kv_heads=2, head_size=d, block_size=64, dtype=dtype,
                                     causal=True, poison=False)
    prob.v_cache.fill_(1.0)
    out = gpu_prefill(prob).float().cpu().numpy()
    err = np.abs(out - 1.0)
    assert np.all(err <= ulp_of(np.ones(1), dtype)[0]), float(err.max())


@pytest.mark.parametrize("rounding", [0, 1, 2])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_first_causal_row_is_v0(rounding, d):
    prob = attn_inputs.paged_problem(seed=42, q_lens=[200, 129], kv_lens=[200, 129],
                                     num_q_heads=8, num_kv_heads=2, head_size=d, block_size=16,
                                     causal=True)
    out = gpu_prefill(prob, rounding=rounding).cpu()
    G = prob.num_q_heads // prob.num_kv_heads
    for b in range(prob.num_seqs):
        t0 = int(prob.query_start_loc[b])
        page = int(prob.block_table[b, 0])
        v0 = prob.v_cache[page, 0]                        # [Hkv, d]: key 0 of sequence b
        for h in range(prob.num_q_heads):
            assert torch.equal(out[t0, h].view(torch.int16), v0[h // G].view(torch.int16)), (b, h)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_decode_split_count_does_not_matter(d):
    prob = attn_inputs.paged_problem(seed=43, q_lens=[1] * 6, kv_lens=[1, 50, 999, 4096, 0, 300],
                                     num_q_heads=16, num_kv_heads=4, head_size=d, block_size=16,
                                     causal=False)
    t = to_dev(prob)
    one = gpu_decode(prob, t=t, splits=1).float().cpu()
    eight = gpu_decode(prob, t=t, splits=8).float().cpu()
    assert float((one - eight).abs().max()) <= TOL[prob.dtype]


def test_outputs_lie_in_the_convex_hull_of_visible_values():
    prob = attn_inputs.paged_problem(seed=44, q_lens=[257, 64], kv_lens=[257, 400], num_q_heads=4,
                                     num_kv_heads=4, head_size=128, block_size=64, causal=True)
    out = gpu_prefill(prob).float().cpu().numpy()
    qsl = prob.query_start_loc.numpy()
    for b in range(prob.num_seqs):
        sq, sk = qsl[b + 1] - qsl[b], prob.kv_lens[b]
        pages = prob.block_table[b, : (sk + 63) // 64].long()
        v = prob.v_cache[pages].reshape(-1, prob.num_kv_heads, 128)[:sk].float().numpy()
        for i in range(sq):
            vis = i + sk - sq + 1                       # keys 0 .. i + Sk - Sq
            lo, hi = v[:vis].min(axis=0), v[:vis].max(axis=0)   # [H, d]
            o = out[qsl[b] + i]
            slack = ulp_of(np.maximum(np.abs(lo), np.abs(hi)), prob.dtype)
            assert np.all(o >= lo - slack) and np.all(o <= hi + slack), (b, i)

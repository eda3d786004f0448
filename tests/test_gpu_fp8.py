"""GPU parity of fp8 K/V caches (E4M3 codes with per-tensor K and V factors;
"gfx942 unified attention, from the math up" sec. 9 lists fp8 among the
feature flags, the convention is stated in include/attn_fwd.h) against the
fp64 oracle, for paged prefill (head sizes 64, 128, 256; the E4M3 pages are
widened into the caller's workspace first) and decode (one and several
splits; the kernels read the codes).

Tolerance: 2e-2 (fp16) / 4e-2 (bf16) max |err|, as for 16-bit caches.  Every
E4M3 value is exact in bf16 and fp16, so with a V factor of 1 the fp8 call
must equal, bit for bit, the 16-bit call on a cache holding the same values
with tau multiplied by the K factor: that ties the fp8 reads to the 16-bit
path exactly.
"""
import numpy as np
import pytest
import torch

import attn_inputs
from oracle import oracle
from tests.helpers import TOL, as_rows, max_err, to_dev, worst

pytestmark = pytest.mark.gpu

F8 = torch.float8_e4m3fn


def problem(seed, d, hq, hkv, bs, dtype=torch.bfloat16, causal=True, q_lens=(300, 1, 129),
            kv_lens=(300, 513, 129)):
    return attn_inputs.paged_problem(seed=seed, q_lens=list(q_lens), kv_lens=list(kv_lens),
                                     num_q_heads=hq, num_kv_heads=hkv, head_size=d,
                                     block_size=bs, dtype=dtype, causal=causal, sigma=1.0,
                                     pool_extra=3, kv_dtype=F8)


def oracle_fp8(prob, **feat):
    return oracle.sdpa(prob.q, prob.k_cache, prob.v_cache, prob.block_table,
                       prob.query_start_loc, prob.seq_lens, num_q_heads=prob.num_q_heads,
                       num_kv_heads=prob.num_kv_heads, head_size=prob.head_size,
                       block_size=prob.block_size, scale=prob.scale, causal=prob.causal,
                       dtype=oracle.BF16 if prob.dtype == torch.bfloat16 else oracle.F16,
                       kv_scales=(prob.k_scale, prob.v_scale), **feat)


def run_prefill(prob, kv_scales=None, t=None, scale=None, **feat):
    import attention_forward_sdpa_gb300 as attn
    t = t or to_dev(prob)
    return attn.prefill(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                        t["query_start_loc"], t["seq_lens"], max_seqlen_q=prob.max_seqlen_q,
                        max_seqlen_k=prob.max_seqlen_k,
                        scale=prob.scale if scale is None else scale, causal=prob.causal,
                        return_lse=True,
                        kv_scales=(prob.k_scale, prob.v_scale) if kv_scales is None else kv_scales,
                        **feat)


def run_decode(prob, splits, kv_scales=None, t=None, scale=None, **feat):
    import attention_forward_sdpa_gb300 as attn
    t = t or to_dev(prob)
    return attn.decode(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"],
                       max_seqlen_k=prob.max_seqlen_k,
                       scale=prob.scale if scale is None else scale, num_splits=splits,
                       return_lse=True,
                       kv_scales=(prob.k_scale, prob.v_scale) if kv_scales is None else kv_scales,
                       **feat)


def check(out, lse, ref, ref_lse, dtype):
    torch.cuda.synchronize()
    got = as_rows(out)
    err = max_err(got, ref)
    assert err <= TOL[dtype], (err, worst(got, ref))
    g = lse.cpu().numpy().reshape(-1).astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(g), fin)
    assert np.max(np.abs(g[fin] - ref_lse[fin])) < 2e-3


SHAPES = {
    # d, Hq, Hkv, block size, dtype
    "d128_gqa4_bf16": (128, 8, 2, 64, torch.bfloat16),
    "d128_mha_fp16": (128, 4, 4, 16, torch.float16),
    "d64_gqa3_bf16": (64, 6, 2, 32, torch.bfloat16),
    "d256_gqa2_bf16": (256, 4, 2, 128, torch.bfloat16),
}


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_fp8(shape, causal):
    d, hq, hkv, bs, dtype = SHAPES[shape]
    prob = problem(91, d, hq, hkv, bs, dtype, causal)
    out, lse = run_prefill(prob)
    check(out, lse, *oracle_fp8(prob), dtype)


@pytest.mark.parametrize("d,hq,hkv", [(128, 32, 8), (128, 16, 2), (64, 6, 2), (256, 8, 2)])
@pytest.mark.parametrize("splits", [1, 8])
def test_decode_fp8(d, hq, hkv, splits):
    prob = problem(92, d, hq, hkv, 16, causal=False, q_lens=[1] * 6,
                   kv_lens=[1, 17, 0, 300, 2049, 700])
    out, lse = run_decode(prob, splits)
    check(out, lse, *oracle_fp8(prob), prob.dtype)


def slopes(h):
    return torch.tensor([2.0 ** (-8.0 * (i + 1) / h) for i in range(h)], dtype=torch.float32)


@pytest.mark.parametrize("kind", ["prefill", "decode"])
def test_fp8_with_score_features(kind):
    hq = 8
    sinks = torch.randn(hq, generator=torch.Generator().manual_seed(3)) * 2.0
    feat = dict(window=(200, -1), softcap=20.0, alibi_slopes=slopes(hq) * 0.1, sinks=sinks)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in feat.items()}
    ofeat = dict(window=feat["window"], softcap=feat["softcap"],
                 alibi_slopes=feat["alibi_slopes"].double().numpy(),
                 sinks=sinks.double().numpy())
    if kind == "prefill":
        prob = problem(93, 128, hq, 2, 64)
        out, lse = run_prefill(prob, **dev)
    else:
        prob = problem(94, 128, hq, 2, 16, causal=False, q_lens=[1] * 4,
                       kv_lens=[700, 33, 1500, 250])
        out, lse = run_decode(prob, 8, **dev)
    check(out, lse, *oracle_fp8(prob, **ofeat), prob.dtype)


def widened(prob):
    """The same problem with bf16 / fp16 caches holding the E4M3 values (exact)."""
    return attn_inputs.PagedProblem(**{**prob.__dict__,
                                       "k_cache": prob.k_cache.to(torch.float32).to(prob.dtype),
                                       "v_cache": prob.v_cache.to(torch.float32).to(prob.dtype),
                                       "k_scale": 1.0, "v_scale": 1.0})


@pytest.mark.parametrize("kind", ["prefill", "decode_tc", "decode_simt"])
def test_unit_v_factor_equals_the_16bit_call_bitwise(kind):
    import attention_forward_sdpa_gb300 as attn
    if kind == "prefill":
        prob = problem(95, 128, 8, 2, 64)
    else:
        d, hq, hkv = (128, 32, 8) if kind == "decode_tc" else (64, 6, 2)
        prob = problem(96, d, hq, hkv, 16, causal=False, q_lens=[1] * 5,
                       kv_lens=[900, 17, 4000, 300, 64])
    w = widened(prob)
    ks = 0.5                      # a power of two: tau * ks is exact on both sides
    if kind == "prefill":
        got, glse = run_prefill(prob, kv_scales=(ks, 1.0))
        t = to_dev(w)
        ref, rlse = attn.prefill(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                 t["query_start_loc"], t["seq_lens"],
                                 max_seqlen_q=w.max_seqlen_q, max_seqlen_k=w.max_seqlen_k,
                                 scale=w.scale * ks, causal=w.causal, return_lse=True)
    else:
        got, glse = run_decode(prob, 8, kv_scales=(ks, 1.0))
        t = to_dev(w)
        ref, rlse = attn.decode(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                t["seq_lens"], max_seqlen_k=w.max_seqlen_k, scale=w.scale * ks,
                                num_splits=8, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(glse, rlse)


def test_fp8_prefill_reports_a_bad_page():
    prob = problem(97, 128, 8, 2, 64)
    t = to_dev(prob)
    t["block_table"][1, 2] = 10_000_000           # referenced by sequence 1 (513 keys)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    import attention_forward_sdpa_gb300 as attn
    attn.prefill(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["query_start_loc"],
                 t["seq_lens"], max_seqlen_q=prob.max_seqlen_q, max_seqlen_k=prob.max_seqlen_k,
                 scale=prob.scale, causal=True, status=status,
                 kv_scales=(prob.k_scale, prob.v_scale))
    torch.cuda.synchronize()
    assert int(status.item()) == 5


@pytest.mark.parametrize("layout", ["bshd", "bhsd", "bshd_padded"])
def test_dense_fp8(layout):
    """fp8 K/V on the dense strided entry point: against the oracle, and bit
    for bit against the paged call on the same codes (one page per batch
    entry)."""
    import attention_forward_sdpa_gb300 as attn
    B, Sq, Sk, hq, hkv, d = 2, 200, 384, 8, 2, 128   # Sk: also a valid paged block size
    prob = attn_inputs.paged_problem(seed=98, q_lens=[Sq] * B, kv_lens=[Sk] * B, num_q_heads=hq,
                                     num_kv_heads=hkv, head_size=d, block_size=Sk, causal=True,
                                     permute=False, poison=False, kv_dtype=F8)
    ks = (prob.k_scale, prob.v_scale)
    q = prob.q.view(B, Sq, hq, d).cuda()
    k = prob.k_cache.view(B, Sk, hkv, d).cuda()
    v = prob.v_cache.view(B, Sk, hkv, d).cuda()
    lay = "bhsd" if layout == "bhsd" else "bshd"
    if layout == "bhsd":
        q, k, v = (x.transpose(1, 2).contiguous() for x in (q, k, v))
    elif layout == "bshd_padded":
        def pad(x, extra):
            big = torch.zeros(*x.shape[:3], x.shape[3] + extra, dtype=x.dtype, device="cuda")
            big[..., :x.shape[3]] = x
            return big[..., :x.shape[3]]
        q, k, v = pad(q, 8), pad(k, 16), pad(v, 32)   # row strides stay 16-byte multiples
    out = attn.dense(q, k, v, layout=lay, scale=prob.scale, causal=True, kv_scales=ks)
    torch.cuda.synchronize()
    packed = (out if lay == "bshd" else out.transpose(1, 2)).contiguous().view(B * Sq, hq, d)
    ref, _ = oracle_fp8(prob)
    got = as_rows(packed)
    assert max_err(got, ref) <= TOL[prob.dtype], worst(got, ref)
    paged, _ = run_prefill(prob)
    torch.cuda.synchronize()
    assert torch.equal(packed.view(torch.int16), paged.view(torch.int16))


# ----------------------------------------------------------------------------
# E4M3 NaN codes (S.1111.111) in positions the kernels read and use
# ----------------------------------------------------------------------------

def _poke(cache, prob, b, j, kvh, c, code=0x7F):
    """Store `code` as channel c of key j (sequence b, KV head kvh)."""
    page = int(prob.block_table[b, j // prob.block_size])
    cache.view(torch.uint8)[page, j % prob.block_size, kvh, c] = code


def _nan_compare(out, lse, ref, ref_lse, dtype, allowed_extra=None):
    """NaN placement and finite values against the oracle.  Every oracle NaN
    must be a kernel NaN.  A kernel NaN the oracle does not have must satisfy
    `allowed_extra(row, channel)` (None: none allowed).  Elements finite on
    both sides agree within the tolerance; so do the finite log-sum-exps."""
    torch.cuda.synchronize()
    got = as_rows(out)
    gn, rn = np.isnan(got), np.isnan(ref)
    assert rn.any(), "the poked codes must reach the oracle's output"
    assert not (rn & ~gn).any(), np.argwhere(rn & ~gn)[:5]
    extra = np.argwhere(gn & ~rn)
    if allowed_extra is None:
        assert extra.size == 0, extra[:5]
    else:
        bad = [tuple(e) for e in extra if not allowed_extra(int(e[0]), int(e[1]))]
        assert not bad, bad[:5]
    both = ~gn & ~rn
    assert np.isfinite(got[both]).all()
    err = float(np.max(np.abs(got[both] - ref[both])))
    assert err <= TOL[dtype], err
    g = lse.cpu().numpy().reshape(-1).astype(np.float64)
    assert not (np.isnan(ref_lse) & ~np.isnan(g)).any()
    fin = np.isfinite(ref_lse) & np.isfinite(g)
    assert np.max(np.abs(g[fin] - ref_lse[fin])) < 2e-3


@pytest.mark.parametrize("d,hq,hkv,splits", [(128, 32, 2, 8), (128, 32, 2, 1), (64, 6, 2, 8),
                                             (128, 6, 2, 4)])
def test_decode_nan_codes_exact_placement(d, hq, hkv, splits):
    """Decode items that hold one KV head (group of 16) and the SIMT kernel's
    shapes (group of 3): a NaN key makes its sequence's rows of that KV head
    NaN, a NaN value element makes that channel NaN, exactly as the
    definition does."""
    prob = problem(120, d, hq, hkv, 16, causal=False, q_lens=[1] * 4,
                   kv_lens=[700, 33, 1500, 250])
    _poke(prob.k_cache, prob, b=0, j=411, kvh=1, c=3)       # a visible key
    _poke(prob.v_cache, prob, b=2, j=1499, kvh=0, c=d - 1)  # the last visible key
    _poke(prob.v_cache, prob, b=3, j=0, kvh=1, c=0, code=0xFF)
    out, lse = run_decode(prob, splits)
    _nan_compare(out, lse, *oracle_fp8(prob), prob.dtype)


def test_decode_nan_value_reaches_the_kv_heads_of_its_item():
    """Group of 4 folds four KV heads into one tcgen05 item: a NaN value of
    one head also reaches, through 0 * NaN in the shared product, that
    channel of the item's other heads (same sequence), and nothing else."""
    hq, hkv, d = 32, 8, 128
    prob = problem(121, d, hq, hkv, 16, causal=False, q_lens=[1] * 3, kv_lens=[900, 2049, 64])
    _poke(prob.k_cache, prob, b=1, j=2000, kvh=5, c=9)
    _poke(prob.v_cache, prob, b=0, j=17, kvh=2, c=77)
    g = hq // hkv

    def allowed(row, ch):        # rows are (sequence, query head)
        b, h = divmod(row, hq)
        return b == 0 and ch == 77 and h // g // 4 == 2 // 4
    out, lse = run_decode(prob, 8)
    _nan_compare(out, lse, *oracle_fp8(prob), prob.dtype, allowed)


def test_prefill_nan_codes():
    """Prefill: a NaN key is exact (masked scores are replaced, not
    multiplied).  A NaN value element of key j reaches that channel in the
    rows of the sequence that see j (the definition) and, through 0 * NaN in
    P.V, the rows of a 128-row query tile that multiplies key j's 128-key
    tile without seeing key j -- nothing else."""
    hq, hkv, d = 8, 2, 128
    prob = problem(122, d, hq, hkv, 64, q_lens=(300, 1, 129), kv_lens=(300, 513, 129))
    _poke(prob.k_cache, prob, b=0, j=5, kvh=0, c=100)       # seen by rows 5.. of sequence 0
    _poke(prob.k_cache, prob, b=1, j=512, kvh=1, c=0)       # the decode-like row's last key
    jv, cv = 200, 31
    _poke(prob.v_cache, prob, b=0, j=jv, kvh=1, c=cv, code=0xFF)
    g = hq // hkv

    def allowed(row, ch):
        tok, h = divmod(row, hq)
        if ch != cv or h // g != 1 or not (0 <= tok < 300):
            return False
        i = tok                              # sequence 0: Sq = Sk = 300, offset 0
        # row i does not see key jv, but its query tile's key loop reaches jv's tile
        return i < jv and (i // 128) * 128 + 127 >= (jv // 128) * 128
    out, lse = run_prefill(prob)
    _nan_compare(out, lse, *oracle_fp8(prob), prob.dtype, allowed)


def test_noncausal_prefill_nan_value_exact():
    """Non-causal: every row multiplies every key it sees and sees every key,
    so a NaN value element gives exactly the definition's NaN channel."""
    prob = problem(123, 128, 4, 2, 64, causal=False, q_lens=(200, 64), kv_lens=(300, 70))
    _poke(prob.v_cache, prob, b=0, j=299, kvh=1, c=64)
    _poke(prob.k_cache, prob, b=1, j=3, kvh=0, c=0)
    out, lse = run_prefill(prob)
    _nan_compare(out, lse, *oracle_fp8(prob), prob.dtype)

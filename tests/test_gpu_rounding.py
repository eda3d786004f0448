"""The epilogue's fp32 -> bf16/fp16 rounding (RTNE, RTNA, RTZ) on the GPU,
through attn_round_f32, against the oracle's rounding (itself pinned to
hand-derived cases, torch casts and a brute-force nearest search): every one
of the 2^32 binary32 patterns in each mode, plus exact ties around random
values."""
import numpy as np
import pytest
import torch

import attention_forward_sdpa_gb300 as attn
from oracle import oracle

pytestmark = pytest.mark.gpu


def patterns():
    bits = np.arange(0, 2**32, 257, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    rng = np.random.default_rng(5)
    out = [x]
    for tdt in (torch.bfloat16, torch.float16):
        lim = 0x7F7F if tdt == torch.bfloat16 else 0x7BFF
        base = rng.integers(1, lim, size=200000).astype(np.uint16)
        lo = torch.from_numpy(base.view(np.int16)).view(tdt).double().numpy()
        hi = torch.from_numpy((base + 1).view(np.int16)).view(tdt).double().numpy()
        mid = ((lo + hi) / 2).astype(np.float32)
        out += [mid, -mid, np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(0))]
    out.append(np.array([0.0, -0.0, np.inf, -np.inf, 65504.0, 65520.0, -65520.0, 1e6,
                         3.4028235e38], dtype=np.float32))
    return np.concatenate(out).astype(np.float32)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_round_matches_oracle(dtype, mode):
    x = patterns()
    xd = torch.from_numpy(x).cuda()
    out = torch.empty(x.size, dtype=torch.int16, device="cuda")
    attn.attn_round_f32(out, xd, dtype=dtype, rounding=mode)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)
    exp = oracle.round_f32(x, oracle.BF16 if dtype == torch.bfloat16 else oracle.F16, mode)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], exp[~nan])
    w = oracle.widen16(got[nan], oracle.BF16 if dtype == torch.bfloat16 else oracle.F16)
    assert np.all(np.isnan(w))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_round_all_binary32_patterns(dtype):
    """Every one of the 2^32 binary32 patterns, in each of the three modes,
    against the oracle's rounding (computed on all host cores, chunk by
    chunk).  NaN inputs must give a NaN of the target format (the payload is
    not specified)."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    odt = oracle.BF16 if dtype == torch.bfloat16 else oracle.F16
    chunk = 1 << 26
    threads = max(1, os.cpu_count() or 1)
    out = torch.empty(chunk, dtype=torch.int16, device="cuda")
    with ThreadPoolExecutor(threads) as pool:
        for mode in (0, 1, 2):
            for start in range(0, 1 << 32, chunk):
                idx = torch.arange(start, start + chunk, dtype=torch.int64, device="cuda")
                bits = torch.where(idx >= (1 << 31), idx - (1 << 32), idx).to(torch.int32)
                attn.attn_round_f32(out, bits.view(torch.float32), dtype=dtype, rounding=mode)
                got = out.cpu().numpy().view(np.uint16)
                x = np.arange(start, start + chunk, dtype=np.uint64).astype(np.uint32).view(np.float32)
                parts = np.array_split(x, threads)
                exp = np.concatenate(list(pool.map(lambda a: oracle.round_f32(a, odt, mode), parts)))
                nan = np.isnan(x)
                bad = np.nonzero((got != exp) & ~nan)[0]
                assert bad.size == 0, (mode, hex(start + int(bad[0])), hex(got[bad[0]]), hex(exp[bad[0]]))
                if nan.any():
                    assert np.all(np.isnan(oracle.widen16(got[nan], odt))), (mode, start)

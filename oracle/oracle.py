"""Python face of the fp64 CPU oracle (sdpa_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg use it; the product package never imports it.  It shares no code
with the CUDA library.  Inputs are the 16-bit tensors (torch CPU tensors or
numpy uint16 arrays) produced by ``attn_inputs``; every arithmetic step runs
in binary64 inside sdpa_oracle.c.

Page citations:
  [ALG] "gfx942 unified attention, from the math up"
  [RDM] "gfx942 unified attention - parity + benchmark harness"
  [MM]  "MoonMath.ai abre un nucleo de atencion HIP para AMD MI300X ..." (7minutos.es)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdpa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libsdpa_oracle.so")

F16, BF16 = 0, 1
RTNE, RTNA, RTZ = 0, 1, 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile sdpa_oracle.c with gcc into oracle/_build (portable flags only)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_sdpa_run.restype = ctypes.c_int
        lib.oracle_sdpa_run.argtypes = [P, P, P, P, P, P, i32, P, P, i32, i32, i32,
                                        i32, i32, f64, i32, i32, i32, i32, P, i64, i32]
        lib.oracle_sdpa_run_ex.restype = ctypes.c_int
        lib.oracle_sdpa_run_ex.argtypes = [P, P, P, P, P, P, i32, P, P, i32, i32, i32,
                                           i32, i32, f64, i32, i32, i32, i32, P, i64, i32,
                                           i32, i32, f64, P, P, i32, f64, f64]
        lib.oracle_round_f32.restype = None
        lib.oracle_round_f32.argtypes = [P, P, i64, i32, i32]
        lib.oracle_widen16_array.restype = None
        lib.oracle_widen16_array.argtypes = [P, P, i64, i32]
        lib.oracle_widen8_array.restype = None
        lib.oracle_widen8_array.argtypes = [P, P, i64]
        _lib = lib
        return lib


def _u16(t) -> np.ndarray:
    """16-bit tensor/array -> contiguous numpy uint16 view of its bits."""
    if isinstance(t, np.ndarray):
        a = t
    else:  # torch tensor (CPU)
        import torch
        a = t.detach().contiguous().view(torch.int16).numpy()
    return np.ascontiguousarray(a).view(np.uint16)


def _u8(t) -> np.ndarray:
    """8-bit tensor/array (uint8 or float8) -> contiguous numpy uint8 view of its bits."""
    if isinstance(t, np.ndarray):
        a = t
    else:  # torch tensor (CPU)
        import torch
        a = t.detach().contiguous().view(torch.uint8).numpy()
    return np.ascontiguousarray(a).view(np.uint8)


def _i32(t) -> np.ndarray:
    if not isinstance(t, np.ndarray):
        t = t.detach().cpu().numpy()
    return np.ascontiguousarray(t, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def sdpa(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, *,
         num_q_heads: int, num_kv_heads: int, head_size: int, block_size: int,
         scale: float, causal: bool, dtype: int, rows=None, variant: int = 0,
         param: int = 0, n_threads: int | None = None, want_lse: bool = True,
         window=(-1, -1), softcap: float = 0.0, alibi_slopes=None, sinks=None,
         kv_scales=None):
    """fp64 SDPA over the paged problem.

    Returns (out, lse): out is float64 [n_rows, head_size] with rows in
    (token, head) order (n_rows = total_q * num_q_heads) or, when ``rows`` is
    given, in the order of the row ids ``token * num_q_heads + head``; lse is
    float64 [n_rows] (natural log), -inf for rows with no visible key.

    variant 0 = definition ([ALG] sec. 1, 2, 4, 5, 10); 1 = online recurrence
    with tile width ``param`` ([ALG] sec. 3); 2 = ``param``-way split with a
    log-sum-exp combine ([ALG] sec. 8).

    Feature flags (variant 0 only; named in [ALG] sec. 9, defined in
    sdpa_oracle.c): ``window`` = (left, right) sliding window around the
    aligned key (-1 = unbounded), ``softcap`` > 0 caps the scaled score at
    c * tanh(s / c), ``alibi_slopes`` [Hq] adds -a_h * |diag - j|, ``sinks``
    [Hq] adds e^(z_h) to the softmax denominator.

    ``kv_scales`` = (k_scale, v_scale) marks the caches as fp8 E4M3 bytes
    (uint8 or float8_e4m3fn tensors): K = k_scale * e4m3(k), V = v_scale *
    e4m3(v); ``dtype`` then names the query / output format only.
    """
    lib = _load()
    qa = _u16(q)
    if kv_scales is None:
        ka, va = _u16(k_cache), _u16(v_cache)
        kv_fp8, k_scale, v_scale = 0, 1.0, 1.0
    else:
        ka, va = _u8(k_cache), _u8(v_cache)
        kv_fp8, k_scale, v_scale = 1, float(kv_scales[0]), float(kv_scales[1])
    bt = _i32(block_table)
    if bt.ndim == 1:
        bt = bt.reshape(1, -1)
    qsl, sl = _i32(query_start_loc), _i32(seq_lens)
    num_seqs = int(sl.shape[0])
    total_q = int(qsl[-1])
    if rows is None:
        n_rows = total_q * num_q_heads
        rows_a = None
    else:
        rows_a = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n_rows = int(rows_a.shape[0])
    out = np.zeros((n_rows, head_size), dtype=np.float64)
    lse = np.zeros((n_rows,), dtype=np.float64) if want_lse else None

    def per_head(x):
        if x is None:
            return None
        if not isinstance(x, np.ndarray):
            x = x.detach().cpu().numpy() if hasattr(x, "detach") else np.asarray(x)
        a = np.ascontiguousarray(x, dtype=np.float64).reshape(-1)
        if a.shape[0] != num_q_heads:
            raise ValueError("per-head feature arrays need num_q_heads entries")
        return a

    al, sk = per_head(alibi_slopes), per_head(sinks)
    rc = lib.oracle_sdpa_run_ex(
        _ptr(out), _ptr(lse) if lse is not None else None,
        _ptr(qa), _ptr(ka), _ptr(va), _ptr(bt), int(bt.shape[1]), _ptr(qsl), _ptr(sl),
        num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
        float(scale), int(bool(causal)), int(dtype), int(variant), int(param),
        _ptr(rows_a) if rows_a is not None else None, n_rows,
        int(n_threads or default_threads()), int(window[0]), int(window[1]), float(softcap),
        _ptr(al) if al is not None else None, _ptr(sk) if sk is not None else None,
        kv_fp8, k_scale, v_scale)
    if rc != 0:
        raise ValueError("oracle rejected the problem description")
    return out, lse


def round_f32(x, dtype: int, mode: int) -> np.ndarray:
    """binary32 values -> uint16 bit patterns of bf16/fp16 in mode RTNE/RTNA/RTZ
    ([MM] "Punto de referencia": nearest-even, nearest ties-away, toward zero)."""
    lib = _load()
    xa = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(xa.shape, dtype=np.uint16)
    lib.oracle_round_f32(_ptr(out), _ptr(xa), int(xa.size), int(dtype), int(mode))
    return out


def widen16(bits, dtype: int) -> np.ndarray:
    """uint16 bit patterns of bf16/fp16 -> exact float64 values."""
    lib = _load()
    a = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    out = np.empty(a.shape, dtype=np.float64)
    lib.oracle_widen16_array(_ptr(out), _ptr(a), int(a.size), int(dtype))
    return out


def widen8(bits) -> np.ndarray:
    """uint8 bit patterns of fp8 E4M3 -> exact float64 values (NaN for S.1111.111)."""
    lib = _load()
    a = np.ascontiguousarray(np.asarray(bits, dtype=np.uint8))
    out = np.empty(a.shape, dtype=np.float64)
    lib.oracle_widen8_array(_ptr(out), _ptr(a), int(a.size))
    return out

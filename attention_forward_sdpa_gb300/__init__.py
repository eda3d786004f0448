"""GB300 (sm_103a) fused scaled-dot-product-attention forward.

Python face of the C ABI in include/attn_fwd.h (libattn_fwd_sm103.so).  This
module only marshals arguments: it checks devices, dtypes and contiguity of
torch tensors, passes raw pointers and sizes, and maps status codes to
exceptions.  Every step of the computation runs in the library's CUDA
kernels; there is no fallback of any kind.  If the library has not been built
(``python -m attention_forward_sdpa_gb300.build_ext``) every call raises.

Entry points (same names as the C functions):
  attn_fwd_prefill, attn_fwd_dense, attn_fwd_decode, attn_fwd_decode_noalloc,
  attn_decode_workspace_size, attn_round_f32, attn_status_string, attn_abi_version
and allocating conveniences ``prefill``, ``dense`` and ``decode`` that create
the output (and the decode workspace) with torch on the inputs' device.

Feature flags (the C calls attn_fwd_prefill_ex / attn_fwd_dense_ex /
attn_fwd_decode_ex, used when any flag is given): ``window=(left, right)``
sliding window around the aligned key (-1 = unbounded), ``softcap`` > 0,
``alibi_slopes`` and ``sinks`` as CUDA fp32 tensors with one entry per query
head.  Their definitions are in include/attn_fwd.h.

fp8 caches: ``kv_scales=(k_scale, v_scale)`` marks ``k_cache`` / ``v_cache``
as torch.float8_e4m3fn (or uint8) tensors of E4M3 codes whose values are
code * k_scale and code * v_scale.  A prefill call then also needs
``fp8_workspace``, a uint8 CUDA tensor of attn_fp8_prefill_workspace_size()
bytes (the allocating ``prefill`` creates it).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import torch

from .build_ext import LIB_PATH

__all__ = ["attn_fwd_prefill", "attn_fwd_dense", "attn_fwd_decode", "attn_fwd_decode_noalloc",
           "has_features", "dense",
           "attn_decode_workspace_size", "attn_fp8_prefill_workspace_size",
           "attn_prefill_split_workspace_size",
           "attn_round_f32", "attn_status_string", "attn_abi_version", "attn_tensor_map_cache_stats",
           "prefill", "decode",
           "AttnError", "library_path", "load_library", "RTNE", "RTNA", "RTZ", "OUT_F32"]

ATTN_OK = 0
STATUS_NAMES = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED",
                3: "ATTN_ERR_CUDA", 4: "ATTN_ERR_WORKSPACE", 5: "ATTN_ERR_BAD_BLOCK_TABLE",
                6: "ATTN_ERR_TIMEOUT"}
F16, BF16 = 0, 1
RTNE, RTNA, RTZ, OUT_F32 = 0, 1, 2, 3

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS_NAMES.get(self.status, self.status)}")


def library_path() -> str:
    return LIB_PATH


def load_library() -> ctypes.CDLL:
    """Loads the built shared library; raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"CUDA library not built: {LIB_PATH} is missing "
                "(run `python -m attention_forward_sdpa_gb300.build_ext`)")
        lib = ctypes.CDLL(LIB_PATH)
        P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                ctypes.c_size_t)
        lib.attn_fwd_prefill.restype = ctypes.c_int
        lib.attn_fwd_prefill.argtypes = [P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32,
                                         i32, i32, i32, f32, i32, ctypes.c_int, ctypes.c_int, P,
                                         P, P]
        lib.attn_fwd_prefill_split.restype = ctypes.c_int
        lib.attn_fwd_prefill_split.argtypes = [P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32,
                                               i32, i32, i32, i32, f32, i32, ctypes.c_int,
                                               ctypes.c_int, P, P, P, sz, P]
        lib.attn_prefill_split_workspace_size.restype = sz
        lib.attn_prefill_split_workspace_size.argtypes = [i32]
        lib.attn_fwd_dense.restype = ctypes.c_int
        lib.attn_fwd_dense.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32,
                                       i32, ctypes.c_int, ctypes.c_int, P, P, P]
        lib.attn_test_prefill_timeout.restype = ctypes.c_int
        lib.attn_test_prefill_timeout.argtypes = [P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32,
                                                  i32, i32, i32, i32, f32, i32, ctypes.c_int,
                                                  ctypes.c_int, P, ctypes.c_uint64, P]
        lib.attn_decode_workspace_size.restype = sz
        lib.attn_decode_workspace_size.argtypes = [i32, i32, i32, i32]
        lib.attn_fp8_prefill_workspace_size.restype = sz
        lib.attn_fp8_prefill_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        lib.attn_fwd_decode.restype = ctypes.c_int
        lib.attn_fwd_decode.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32,
                                        f32, i32, ctypes.c_int, ctypes.c_int, P, P, sz, P, P]
        lib.attn_fwd_decode_noalloc.restype = ctypes.c_int
        lib.attn_fwd_decode_noalloc.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32,
                                                i32, i32, f32, i32, ctypes.c_int, ctypes.c_int, P,
                                                P, P]
        FP = ctypes.POINTER(_Features)
        lib.attn_fwd_prefill_ex.restype = ctypes.c_int
        lib.attn_fwd_prefill_ex.argtypes = list(lib.attn_fwd_prefill.argtypes) + [FP]
        lib.attn_fwd_dense_ex.restype = ctypes.c_int
        lib.attn_fwd_dense_ex.argtypes = list(lib.attn_fwd_dense.argtypes) + [FP]
        lib.attn_fwd_decode_ex.restype = ctypes.c_int
        lib.attn_fwd_decode_ex.argtypes = list(lib.attn_fwd_decode.argtypes) + [FP]
        lib.attn_round_f32.restype = ctypes.c_int
        lib.attn_round_f32.argtypes = [P, P, i64, ctypes.c_int, ctypes.c_int, P]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_status_string.argtypes = [ctypes.c_int]
        lib.attn_abi_version.restype = i32
        lib.attn_abi_version.argtypes = []
        lib.attn_tensor_map_cache_stats.restype = None
        lib.attn_tensor_map_cache_stats.argtypes = [P, P]
        _lib = lib
        return lib


# ----------------------------------------------------------------------------
# marshalling helpers
# ----------------------------------------------------------------------------

def _dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return BF16
    if t == torch.float16:
        return F16
    raise TypeError(f"unsupported dtype {t}: expected torch.bfloat16 or torch.float16")


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _same_device(dev, **tensors):
    """Every given tensor on `dev` (the query's device): the library launches
    on the current device, which the calls below set to `dev`."""
    idx = dev.index
    for name, t in tensors.items():
        if t is not None and t.get_device() != idx:
            raise ValueError(f"{name} is on {t.device}, q on {dev}")


def _on(dev):
    """Makes `dev` the current device for the call (no switch when it is)."""
    if dev.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(dev)


def _check_out_arrays(lse, lse_shape, status):
    """lse (when given) holds exactly one fp32 per (row, head); status (when
    given) at least one int32 word."""
    if lse is not None and tuple(lse.shape) != tuple(lse_shape):
        raise ValueError(f"lse must have shape {tuple(lse_shape)}, got {tuple(lse.shape)}")
    if status is not None and status.numel() < 1:
        raise ValueError("status must hold at least one int32 word")


def _dims(t, n, name):
    if t.dim() != n:
        raise ValueError(f"{name} must be {n}-D, got {t.dim()}-D")


def _stream_handle(stream) -> ctypes.c_void_p:
    """The cudaStream_t of `stream` (None: the current stream of the current
    device, which the calls set to the query's device).  A torch stream must
    belong to that device; a raw handle is passed through as given."""
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        if stream.device.index != torch.cuda.current_device():
            raise ValueError(f"stream is on {stream.device}, the call on "
                             f"cuda:{torch.cuda.current_device()}")
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(rc: int, where: str):
    if rc != ATTN_OK:
        raise AttnError(rc, where)


class _Features(ctypes.Structure):
    """attn_features_t"""
    _fields_ = [("window_left", ctypes.c_int32), ("window_right", ctypes.c_int32),
                ("softcap", ctypes.c_float), ("alibi_slopes", ctypes.c_void_p),
                ("sinks", ctypes.c_void_p), ("kv_fp8", ctypes.c_int32),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


def _features(num_q_heads: int, window=None, softcap: float = 0.0, alibi_slopes=None,
              sinks=None, kv_scales=None, fp8_workspace=None):
    """The attn_features_t of a call, or None for a plain call."""
    if not has_features(window, softcap, alibi_slopes, sinks, kv_scales):
        return None
    wl, wr = (-1, -1) if window is None else (int(window[0]), int(window[1]))
    for t, name in ((alibi_slopes, "alibi_slopes"), (sinks, "sinks")):
        if t is not None:
            _dev(t, name, torch.float32)
            if t.numel() != num_q_heads:
                raise ValueError(f"{name} needs one entry per query head ({num_q_heads})")
    ws, ws_bytes = None, 0
    if fp8_workspace is not None:
        _dev(fp8_workspace, "fp8_workspace")
        ws, ws_bytes = fp8_workspace.data_ptr(), fp8_workspace.numel() * fp8_workspace.element_size()
    ks, vs = (1.0, 1.0) if kv_scales is None else (float(kv_scales[0]), float(kv_scales[1]))
    return _Features(wl, wr, float(softcap),
                     None if alibi_slopes is None else alibi_slopes.data_ptr(),
                     None if sinks is None else sinks.data_ptr(),
                     0 if kv_scales is None else 1, ks, vs, ws, ws_bytes)


def has_features(window=None, softcap: float = 0.0, alibi_slopes=None, sinks=None,
                 kv_scales=None) -> bool:
    """True when a call carries any feature flag."""
    return not (window is None and not softcap and alibi_slopes is None and sinks is None and
                kv_scales is None)


_FP8_CACHE_DTYPES = (torch.float8_e4m3fn, torch.uint8)


def _cache_dev(t, name, q_dtype, kv_scales):
    """A K/V cache: the query dtype, or E4M3 codes when kv_scales is given."""
    if kv_scales is None:
        return _dev(t, name, q_dtype)
    _dev(t, name)
    if t.dtype not in _FP8_CACHE_DTYPES:
        raise TypeError(f"{name} must be torch.float8_e4m3fn or uint8 with kv_scales, got {t.dtype}")


# ----------------------------------------------------------------------------
# C entry points
# ----------------------------------------------------------------------------

def attn_abi_version() -> int:
    return int(load_library().attn_abi_version())


def attn_tensor_map_cache_stats() -> tuple:
    """(hits, misses) of the library's tensor-map cache."""
    h, m = ctypes.c_uint64(0), ctypes.c_uint64(0)
    load_library().attn_tensor_map_cache_stats(ctypes.byref(h), ctypes.byref(m))
    return int(h.value), int(m.value)


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def attn_decode_workspace_size(num_seqs: int, num_q_heads: int, head_size: int,
                               num_splits: int) -> int:
    return int(load_library().attn_decode_workspace_size(num_seqs, num_q_heads, head_size,
                                                         num_splits))


def attn_fp8_prefill_workspace_size(num_seqs: int, max_seqlen_k: int, num_kv_heads: int,
                                    head_size: int, block_size: int) -> int:
    return int(load_library().attn_fp8_prefill_workspace_size(num_seqs, max_seqlen_k,
                                                              num_kv_heads, head_size,
                                                              block_size))


def attn_fwd_prefill(out, q, k_cache, v_cache, block_table, query_start_loc, seq_lens, *,
                     max_seqlen_q: int, max_seqlen_k: int, scale: float, causal: bool,
                     rounding: int = RTNE, lse=None, status=None, stream=None, window=None,
                     softcap: float = 0.0, alibi_slopes=None, sinks=None, kv_scales=None,
                     fp8_workspace=None, split_workspace=None) -> None:
    """Calls attn_fwd_prefill (attn_fwd_prefill_ex with feature flags, or
    attn_fwd_prefill_split when ``split_workspace`` -- a uint8 CUDA tensor of
    attn_prefill_split_workspace_size(head_size) bytes -- is given) on torch
    CUDA tensors (shapes as in the C header)."""
    lib = load_library()
    dt = _dtype_code(q.dtype)
    _dev(q, "q")
    _cache_dev(k_cache, "k_cache", q.dtype, kv_scales)
    _cache_dev(v_cache, "v_cache", q.dtype, kv_scales)
    _dev(out, "out", torch.float32 if rounding == OUT_F32 else q.dtype)
    _dev(block_table, "block_table", torch.int32)
    _dev(query_start_loc, "query_start_loc", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    if lse is not None:
        _dev(lse, "lse", torch.float32)
    if status is not None:
        _dev(status, "status", torch.int32)
    _dims(q, 3, "q")
    _dims(k_cache, 4, "k_cache")
    total_q, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("inconsistent q / k_cache / v_cache / out shapes")
    _dims(seq_lens, 1, "seq_lens")
    num_seqs = seq_lens.shape[0]
    if query_start_loc.dim() != 1 or query_start_loc.shape[0] != num_seqs + 1 or \
            block_table.dim() != 2 or block_table.shape[0] != num_seqs:
        raise ValueError("inconsistent query_start_loc / block_table / seq_lens shapes")
    _check_out_arrays(lse, (total_q, hq), status)
    _same_device(q.device, out=out, k_cache=k_cache, v_cache=v_cache, block_table=block_table,
                 query_start_loc=query_start_loc, seq_lens=seq_lens, lse=lse, status=status,
                 alibi_slopes=alibi_slopes, sinks=sinks, fp8_workspace=fp8_workspace)
    with _on(q.device):
        args = (_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                block_table.shape[1], _ptr(query_start_loc), _ptr(seq_lens), num_seqs,
                int(max_seqlen_q), int(max_seqlen_k), total_q, hq, hkv, d, bs, nb, float(scale),
                int(bool(causal)), dt, int(rounding), _ptr(lse), _ptr(status),
                _stream_handle(stream))
        feat = _features(hq, window, softcap, alibi_slopes, sinks, kv_scales, fp8_workspace)
        if split_workspace is not None:
            if feat is not None:
                raise ValueError("the split prefill takes no feature flags")
            _dev(split_workspace, "split_workspace", torch.uint8)
            _same_device(q.device, split_workspace=split_workspace)
            _check(lib.attn_fwd_prefill_split(*args[:-1], _ptr(split_workspace),
                                              split_workspace.numel(), args[-1]),
                   "attn_fwd_prefill_split")
        elif feat is None:
            _check(lib.attn_fwd_prefill(*args), "attn_fwd_prefill")
        else:
            _check(lib.attn_fwd_prefill_ex(*args, ctypes.byref(feat)), "attn_fwd_prefill_ex")


def _strides3(t, name):
    """(batch, sequence, head) element strides of a logical [B, S, H, d] view,
    which may be a permuted view (for instance BHSD memory seen as BSHD)."""
    if t.dim() != 4:
        raise ValueError(f"{name} must be 4-D [batch, seq, heads, head_size]")
    if t.stride(3) != 1:
        raise ValueError(f"{name}: the head_size dimension must be contiguous")
    return (ctypes.c_int64 * 3)(t.stride(0), t.stride(1), t.stride(2))


def attn_fwd_dense(out, q, k, v, *, scale: float, causal: bool, rounding: int = RTNE, lse=None,
                   status=None, stream=None, window=None, softcap: float = 0.0,
                   alibi_slopes=None, sinks=None, kv_scales=None, fp8_workspace=None) -> None:
    """Calls attn_fwd_dense on logical [batch, seq, heads, head_size] CUDA
    tensors in any (batch, seq, head) stride order: BSHD tensors as they are,
    BHSD tensors x as x.transpose(1, 2) (a view, nothing is copied)."""
    lib = load_library()
    dt = _dtype_code(q.dtype)
    kv_want = None if kv_scales is not None else q.dtype
    for t, name, want in ((q, "q", None), (k, "k", kv_want), (v, "v", kv_want),
                          (out, "out", torch.float32 if rounding == OUT_F32 else q.dtype)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if want is not None and t.dtype != want:
            raise TypeError(f"{name} must be {want}, got {t.dtype}")
    if kv_scales is not None:
        for t, name in ((k, "k"), (v, "v")):
            if t.dtype not in _FP8_CACHE_DTYPES:
                raise TypeError(f"{name} must be torch.float8_e4m3fn or uint8 with kv_scales")
    if lse is not None:
        _dev(lse, "lse", torch.float32)
    if status is not None:
        _dev(status, "status", torch.int32)
    qs, ks, vs, os_ = (_strides3(q, "q"), _strides3(k, "k"), _strides3(v, "v"),
                       _strides3(out, "out"))
    b, sq, hq, d = q.shape
    b2, sk, hkv, d2 = k.shape
    if b2 != b or d2 != d or tuple(v.shape) != tuple(k.shape) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("inconsistent q / k / v / out shapes")
    _check_out_arrays(lse, (b, hq, sq), status)
    _same_device(q.device, out=out, k=k, v=v, lse=lse, status=status, alibi_slopes=alibi_slopes,
                 sinks=sinks, fp8_workspace=fp8_workspace)
    with _on(q.device):
        args = (_ptr(out), _ptr(q), _ptr(k), _ptr(v), qs, ks, vs, os_, b, sq, sk, hq, hkv, d,
                float(scale), int(bool(causal)), dt, int(rounding), _ptr(lse), _ptr(status),
                _stream_handle(stream))
        feat = _features(hq, window, softcap, alibi_slopes, sinks, kv_scales, fp8_workspace)
        if feat is None:
            _check(lib.attn_fwd_dense(*args), "attn_fwd_dense")
        else:
            _check(lib.attn_fwd_dense_ex(*args, ctypes.byref(feat)), "attn_fwd_dense_ex")


def attn_fwd_decode(out, q, k_cache, v_cache, block_table, seq_lens, *, max_seqlen_k: int,
                    scale: float, num_splits: int, workspace=None, rounding: int = RTNE,
                    lse=None, status=None, stream=None, window=None, softcap: float = 0.0,
                    alibi_slopes=None, sinks=None, kv_scales=None) -> None:
    """Calls attn_fwd_decode (attn_fwd_decode_ex with feature flags) on torch
    CUDA tensors (shapes as in the C header)."""
    lib = load_library()
    dt = _dtype_code(q.dtype)
    _dev(q, "q")
    _cache_dev(k_cache, "k_cache", q.dtype, kv_scales)
    _cache_dev(v_cache, "v_cache", q.dtype, kv_scales)
    _dev(out, "out", torch.float32 if rounding == OUT_F32 else q.dtype)
    _dev(block_table, "block_table", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    if lse is not None:
        _dev(lse, "lse", torch.float32)
    if status is not None:
        _dev(status, "status", torch.int32)
    ws_bytes = 0
    if workspace is not None:
        _dev(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    _dims(q, 3, "q")
    _dims(k_cache, 4, "k_cache")
    num_seqs, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("inconsistent q / k_cache / v_cache / out shapes")
    if seq_lens.dim() != 1 or seq_lens.shape[0] != num_seqs or block_table.dim() != 2 or \
            block_table.shape[0] != num_seqs:
        raise ValueError("inconsistent block_table / seq_lens shapes")
    _check_out_arrays(lse, (num_seqs, hq), status)
    _same_device(q.device, out=out, k_cache=k_cache, v_cache=v_cache, block_table=block_table,
                 seq_lens=seq_lens, lse=lse, status=status, workspace=workspace,
                 alibi_slopes=alibi_slopes, sinks=sinks)
    with _on(q.device):
        args = (_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                block_table.shape[1], _ptr(seq_lens), num_seqs, int(max_seqlen_k), hq, hkv, d, bs,
                nb, float(scale), int(num_splits), dt, int(rounding), _ptr(lse), _ptr(workspace),
                ws_bytes, _ptr(status), _stream_handle(stream))
        feat = _features(hq, window, softcap, alibi_slopes, sinks, kv_scales)
        if feat is None:
            _check(lib.attn_fwd_decode(*args), "attn_fwd_decode")
        else:
            _check(lib.attn_fwd_decode_ex(*args, ctypes.byref(feat)), "attn_fwd_decode_ex")


def attn_fwd_decode_noalloc(out, q, k_cache, v_cache, block_table, seq_lens, *,
                            max_seqlen_k: int, scale: float, num_splits: int,
                            rounding: int = RTNE, lse=None, status=None, stream=None) -> None:
    """Calls attn_fwd_decode_noalloc: the decode without a caller workspace, for
    callers that may not allocate device memory (the split partials live in a
    library-owned device array of ATTN_DECODE_NOALLOC_SCRATCH_BYTES; calls on
    one device must not overlap)."""
    lib = load_library()
    dt = _dtype_code(q.dtype)
    _dev(q, "q")
    _dev(k_cache, "k_cache", q.dtype)
    _dev(v_cache, "v_cache", q.dtype)
    _dev(out, "out", torch.float32 if rounding == OUT_F32 else q.dtype)
    _dev(block_table, "block_table", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    if lse is not None:
        _dev(lse, "lse", torch.float32)
    if status is not None:
        _dev(status, "status", torch.int32)
    _dims(q, 3, "q")
    _dims(k_cache, 4, "k_cache")
    num_seqs, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("inconsistent q / k_cache / v_cache / out shapes")
    if seq_lens.dim() != 1 or seq_lens.shape[0] != num_seqs or block_table.dim() != 2 or \
            block_table.shape[0] != num_seqs:
        raise ValueError("inconsistent block_table / seq_lens shapes")
    _check_out_arrays(lse, (num_seqs, hq), status)
    _same_device(q.device, out=out, k_cache=k_cache, v_cache=v_cache, block_table=block_table,
                 seq_lens=seq_lens, lse=lse, status=status)
    with _on(q.device):
        rc = lib.attn_fwd_decode_noalloc(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                         _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                                         num_seqs, int(max_seqlen_k), hq, hkv, d, bs, nb,
                                         float(scale), int(num_splits), dt, int(rounding),
                                         _ptr(lse), _ptr(status), _stream_handle(stream))
    _check(rc, "attn_fwd_decode_noalloc")


def attn_round_f32(out, x, *, dtype: torch.dtype, rounding: int, stream=None) -> None:
    """Rounds fp32 CUDA tensor x into out (int16 tensor of the same size holding
    bf16/fp16 bit patterns) with the epilogue's rounding."""
    lib = load_library()
    _dev(x, "x", torch.float32)
    _dev(out, "out")
    if out.element_size() != 2 or out.numel() != x.numel():
        raise ValueError("out must be a 16-bit tensor with as many elements as x")
    _same_device(x.device, out=out)
    with _on(x.device):
        _check(lib.attn_round_f32(_ptr(out), _ptr(x), x.numel(), _dtype_code(dtype),
                                  int(rounding), _stream_handle(stream)), "attn_round_f32")


# ----------------------------------------------------------------------------
# allocating conveniences
# ----------------------------------------------------------------------------

def attn_prefill_split_workspace_size(head_size: int) -> int:
    return int(load_library().attn_prefill_split_workspace_size(int(head_size)))


def prefill(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, *, max_seqlen_q: int,
            max_seqlen_k: int, scale: float | None = None, causal: bool = True,
            rounding: int = RTNE, return_lse: bool = False, status=None, stream=None,
            split: bool = False, **features):
    """Returns O (and the log-sum-exp when asked) for a paged prefill problem.
    ``features``: window, softcap, alibi_slopes, sinks, kv_scales (see the
    module doc); with kv_scales the fp8 workspace is allocated here.
    ``split=True`` runs attn_fwd_prefill_split with a workspace allocated here."""
    if scale is None:
        scale = q.shape[-1] ** -0.5
    out = torch.empty(q.shape, dtype=torch.float32 if rounding == OUT_F32 else q.dtype,
                      device=q.device)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device) if return_lse else None
    if features.get("kv_scales") is not None and features.get("fp8_workspace") is None:
        nbytes = attn_fp8_prefill_workspace_size(seq_lens.shape[0], int(max_seqlen_k),
                                                 k_cache.shape[2], k_cache.shape[3],
                                                 k_cache.shape[1])
        features = dict(features, fp8_workspace=torch.empty(max(nbytes, 1), dtype=torch.uint8,
                                                            device=q.device))
    if split:
        features = dict(features, split_workspace=torch.empty(
            attn_prefill_split_workspace_size(q.shape[-1]), dtype=torch.uint8, device=q.device))
    attn_fwd_prefill(out, q, k_cache, v_cache, block_table, query_start_loc, seq_lens,
                     max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k, scale=scale,
                     causal=causal, rounding=rounding, lse=lse, status=status, stream=stream,
                     **features)
    return (out, lse) if return_lse else out


def dense(q, k, v, *, layout: str = "bshd", scale: float | None = None, causal: bool = False,
          rounding: int = RTNE, return_lse: bool = False, status=None, stream=None, **features):
    """Returns O in the layout of q for fixed-length batches: layout "bshd"
    takes [B, S, H, d] tensors, "bhsd" takes [B, H, S, d] tensors (read in
    place).  The log-sum-exp, when asked, is [B, H, Sq] fp32."""
    if layout not in ("bshd", "bhsd"):
        raise ValueError("layout must be 'bshd' or 'bhsd'")
    if scale is None:
        scale = q.shape[-1] ** -0.5
    out = torch.empty(q.shape, dtype=torch.float32 if rounding == OUT_F32 else q.dtype,
                      device=q.device)
    view = (lambda t: t.transpose(1, 2)) if layout == "bhsd" else (lambda t: t)
    qv = view(q)
    lse = (torch.empty((qv.shape[0], qv.shape[2], qv.shape[1]), dtype=torch.float32,
                       device=q.device) if return_lse else None)
    if features.get("kv_scales") is not None and features.get("fp8_workspace") is None:
        kv = view(k)
        nbytes = attn_fp8_prefill_workspace_size(kv.shape[0], kv.shape[1], kv.shape[2],
                                                 kv.shape[3], max(kv.shape[1], 1))
        features = dict(features, fp8_workspace=torch.empty(max(nbytes, 1), dtype=torch.uint8,
                                                            device=q.device))
    attn_fwd_dense(view(out), qv, view(k), view(v), scale=scale, causal=causal, rounding=rounding,
                   lse=lse, status=status, stream=stream, **features)
    return (out, lse) if return_lse else out


def decode(q, k_cache, v_cache, block_table, seq_lens, *, max_seqlen_k: int,
           scale: float | None = None, num_splits: int = 8, rounding: int = RTNE,
           return_lse: bool = False, workspace=None, status=None, stream=None, **features):
    """Returns O (and the log-sum-exp when asked) for one decode step."""
    if scale is None:
        scale = q.shape[-1] ** -0.5
    out = torch.empty(q.shape, dtype=torch.float32 if rounding == OUT_F32 else q.dtype,
                      device=q.device)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device) if return_lse else None
    if workspace is None:
        n = attn_decode_workspace_size(q.shape[0], q.shape[1], q.shape[2], num_splits)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device) if n else None
    attn_fwd_decode(out, q, k_cache, v_cache, block_table, seq_lens, max_seqlen_k=max_seqlen_k,
                    scale=scale, num_splits=num_splits, workspace=workspace, rounding=rounding,
                    lse=lse, status=status, stream=stream, **features)
    return (out, lse) if return_lse else out

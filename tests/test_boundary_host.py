"""Host-side checks of the C ABI (no GPU needed, nothing is launched).

  - the shared library builds, loads and exports every function that
    include/attn_fwd.h declares, and the header serves a plain C99 program;
  - argument errors are returned before any CUDA call (so they work on a
    machine without a GPU): null pointers, head-group mismatch, head sizes and
    block sizes outside the compiled set, bad enums, bad scale, short block
    table, missing workspace;
  - the workspace size is plain arithmetic;
  - the Python binding refuses CPU tensors and wrong dtypes instead of
    falling back to anything.
"""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    from attention_forward_sdpa_gb300 import build_ext
    import attention_forward_sdpa_gb300 as pkg
    build_ext.build()
    return pkg.load_library()


def declared_functions():
    names = []
    for f in sorted(os.listdir(HEADER_DIR)):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(attn_\w+)\s*\(", text, flags=re.M):
            names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("attn_fwd_prefill", "attn_fwd_dense", "attn_fwd_decode", "attn_decode_workspace_size",
              "attn_round_f32", "attn_status_string", "attn_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings_and_version(lib):
    assert lib.attn_abi_version() == 2
    for code in range(7):
        assert lib.attn_status_string(code)
    assert lib.attn_status_string(99) == b"unknown status"


def test_workspace_size_is_arithmetic(lib):
    assert lib.attn_decode_workspace_size(64, 32, 128, 8) == 64 * 32 * 8 * (128 + 2) * 4 + 256
    assert lib.attn_decode_workspace_size(64, 32, 128, 1) == 256
    assert lib.attn_decode_workspace_size(0, 32, 128, 8) == 0


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first


def prefill_args(**over):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, bt_stride=4, qsl=FAKE, sl=FAKE,
             num_seqs=2, max_q=100, max_k=200, total_q=150, hq=8, hkv=2, d=128, bs=64, nb=10,
             scale=0.088, causal=1, dtype=1, rounding=0, lse=None, status=None, stream=None)
    a.update(over)
    return [a[k] for k in ("out", "q", "k", "v", "bt", "bt_stride", "qsl", "sl", "num_seqs",
                           "max_q", "max_k", "total_q", "hq", "hkv", "d", "bs", "nb", "scale",
                           "causal", "dtype", "rounding", "lse", "status", "stream")]


@pytest.mark.parametrize("over,code", [
    (dict(q=None), 1),
    (dict(out=None), 1),
    (dict(bt=None), 1),
    (dict(hq=6, hkv=4), 1),
    (dict(hkv=0), 1),
    (dict(d=96), 2),
    (dict(d=512), 2),
    (dict(d=32), 2),
    (dict(bs=48), 2),
    (dict(bs=8), 2),
    (dict(bs=192), 2),
    (dict(dtype=7), 1),
    (dict(rounding=9), 1),
    (dict(causal=2), 1),
    (dict(scale=0.0), 1),
    (dict(scale=float("nan")), 1),
    (dict(bt_stride=3), 1),
    (dict(num_seqs=-1), 1),
    (dict(q=ctypes.c_void_p(0x10008)), 1),
    (dict(bt=ctypes.c_void_p(0x10002)), 1),      # int32 / fp32 arrays: 4-byte aligned
    (dict(qsl=ctypes.c_void_p(0x10001)), 1),
    (dict(sl=ctypes.c_void_p(0x10003)), 1),
    (dict(lse=ctypes.c_void_p(0x10002)), 1),
    (dict(status=ctypes.c_void_p(0x10001)), 1),
])
def test_prefill_rejects_bad_arguments(lib, over, code):
    assert lib.attn_fwd_prefill(*prefill_args(**over)) == code


def test_prefill_empty_problem_is_a_no_op(lib):
    assert lib.attn_fwd_prefill(*prefill_args(num_seqs=0)) == 0
    assert lib.attn_fwd_prefill(*prefill_args(total_q=0)) == 0


def split_args(ws=FAKE, ws_bytes=None, **over):
    """attn_fwd_prefill_split: attn_fwd_prefill's arguments with the workspace
    before the stream."""
    a = prefill_args(**over)
    return a[:-1] + [ws, ws_bytes if ws_bytes is not None else 64 << 20, a[-1]]


def test_split_workspace_size(lib):
    lib.attn_prefill_split_workspace_size.restype = ctypes.c_size_t
    lib.attn_prefill_split_workspace_size.argtypes = [ctypes.c_int32]
    n128 = lib.attn_prefill_split_workspace_size(128)
    n64 = lib.attn_prefill_split_workspace_size(64)
    # 2 parts per CTA x 160 CTAs x 2 tiles x 128 rows of (d + 2) fp32, plus the tickets
    assert n128 == (2 * 160 * 2 * 128 * 130 * 4 + 160 * 8 + 255) // 256 * 256
    assert n64 == (2 * 160 * 2 * 128 * 66 * 4 + 160 * 8 + 255) // 256 * 256
    assert lib.attn_prefill_split_workspace_size(80) == 0
    assert n128 % 256 == 0


@pytest.mark.parametrize("over,code", [
    (dict(ws=None), 4),
    (dict(ws_bytes=1024), 4),
    (dict(ws=ctypes.c_void_p(0x10080)), 4),           # not 256-byte aligned
    (dict(q=None), 1),
    (dict(d=80), 2),
    (dict(bs=24), 2),
    (dict(num_seqs=0), 0),
])
def test_split_prefill_rejects_bad_arguments(lib, over, code):
    lib.attn_fwd_prefill_split.restype = ctypes.c_int
    assert lib.attn_fwd_prefill_split(*split_args(**over)) == code


def decode_args(**over):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, bt_stride=512, sl=FAKE, num_seqs=64,
             max_k=8192, hq=32, hkv=8, d=128, bs=16, nb=100000, scale=0.088, splits=8, dtype=1,
             rounding=0, lse=None, ws=FAKE, ws_bytes=64 * 32 * 8 * 130 * 4 + 256, status=None,
             stream=None)
    a.update(over)
    return [a[k] for k in ("out", "q", "k", "v", "bt", "bt_stride", "sl", "num_seqs", "max_k",
                           "hq", "hkv", "d", "bs", "nb", "scale", "splits", "dtype", "rounding",
                           "lse", "ws", "ws_bytes", "status", "stream")]


@pytest.mark.parametrize("over,code", [
    (dict(q=None), 1),
    (dict(sl=None), 1),
    (dict(hq=30), 1),
    (dict(d=80), 2),
    (dict(bs=24), 2),
    (dict(splits=0), 1),
    (dict(splits=65), 1),
    (dict(bt_stride=511), 1),
    (dict(ws=None), 4),
    (dict(ws_bytes=100), 4),
    (dict(ws=ctypes.c_void_p(0x10004)), 4),
    (dict(rounding=4), 1),
    (dict(bt=ctypes.c_void_p(0x10002)), 1),
    (dict(sl=ctypes.c_void_p(0x10001)), 1),
    (dict(lse=ctypes.c_void_p(0x10003)), 1),
    (dict(status=ctypes.c_void_p(0x10002)), 1),
])
def test_decode_rejects_bad_arguments(lib, over, code):
    assert lib.attn_fwd_decode(*decode_args(**over)) == code


@pytest.mark.parametrize("over,code", [
    (dict(q=None), 1),
    (dict(q=ctypes.c_void_p(0x10008)), 1),
    (dict(bt=ctypes.c_void_p(0x10002)), 1),
    (dict(sl=ctypes.c_void_p(0x10001)), 1),
    (dict(lse=ctypes.c_void_p(0x10003)), 1),
    (dict(status=ctypes.c_void_p(0x10002)), 1),
    (dict(d=80), 2),
    (dict(splits=65), 1),
    (dict(num_seqs=0), 0),
])
def test_noalloc_decode_rejects_bad_arguments(lib, over, code):
    a = decode_args(**over)
    del a[19:21]                                  # no workspace arguments
    assert lib.attn_fwd_decode_noalloc(*a) == code


S3 = (ctypes.c_int64 * 3)


def dense_args(**over):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, qs=S3(4096, 1024, 128), ks=S3(4096, 256, 128),
             vs=S3(4096, 256, 128), os=S3(4096, 1024, 128), b=2, sq=32, sk=16, hq=8, hkv=2, d=128,
             scale=0.088, causal=1, dtype=1, rounding=0, lse=None, status=None, stream=None)
    a.update(over)
    return [a[k] for k in ("out", "q", "k", "v", "qs", "ks", "vs", "os", "b", "sq", "sk", "hq",
                           "hkv", "d", "scale", "causal", "dtype", "rounding", "lse", "status",
                           "stream")]


@pytest.mark.parametrize("over,code", [
    (dict(q=None), 1),
    (dict(out=None), 1),
    (dict(qs=None), 1),
    (dict(os=None), 1),
    (dict(ks=S3(4096, 256, 0)), 1),          # zero stride
    (dict(vs=S3(4096, -256, 128)), 1),       # negative stride
    (dict(qs=S3(4096, 1020, 128)), 1),       # 2040 bytes: not a multiple of 16
    (dict(os=S3(4096, 1024, 130), rounding=3), 1),
    (dict(hq=6, hkv=4), 1),
    (dict(d=96), 2),
    (dict(dtype=5), 1),
    (dict(rounding=7), 1),
    (dict(causal=3), 1),
    (dict(scale=-1.0), 1),
    (dict(b=-1), 1),
    (dict(q=ctypes.c_void_p(0x10008)), 1),
    (dict(lse=ctypes.c_void_p(0x10002)), 1),
    (dict(status=ctypes.c_void_p(0x10001)), 1),
])
def test_dense_rejects_bad_arguments(lib, over, code):
    assert lib.attn_fwd_dense(*dense_args(**over)) == code


def test_dense_empty_problem_is_a_no_op(lib):
    assert lib.attn_fwd_dense(*dense_args(b=0)) == 0
    assert lib.attn_fwd_dense(*dense_args(sq=0)) == 0


def test_timeout_hook_rejects_bad_arguments(lib):
    a = prefill_args()
    a.pop(21)   # the hook has no lse argument
    status = ctypes.c_void_p(0x20000)
    stream = a.pop()
    a.pop()     # status
    assert lib.attn_test_prefill_timeout(*a, None, 20_000_000, stream) == 1        # status required
    assert lib.attn_test_prefill_timeout(*a, status, 999, stream) == 1             # limit < 1 ms
    assert lib.attn_test_prefill_timeout(*a, status, 5_000_000_000, stream) == 1   # limit > 4 s


class Feat(ctypes.Structure):
    _fields_ = [("window_left", ctypes.c_int32), ("window_right", ctypes.c_int32),
                ("softcap", ctypes.c_float), ("alibi_slopes", ctypes.c_void_p),
                ("sinks", ctypes.c_void_p)]


@pytest.mark.parametrize("feat", [
    Feat(-2, -1, 0.0, None, None),                 # window below -1
    Feat(-1, -5, 0.0, None, None),
    Feat(-1, -1, -1.0, None, None),                # negative softcap
    Feat(-1, -1, float("nan"), None, None),
    Feat(-1, -1, float("inf"), None, None),
    Feat(-1, -1, 0.0, 0x10002, None),              # misaligned per-head arrays
    Feat(-1, -1, 0.0, None, 0x10001),
])
def test_feature_flags_are_validated(lib, feat):
    import attention_forward_sdpa_gb300 as pkg
    pkg.load_library()                             # sets the _ex argtypes
    P = ctypes.POINTER(pkg._Features)
    f = pkg._Features(feat.window_left, feat.window_right, feat.softcap, feat.alibi_slopes,
                      feat.sinks)
    assert lib.attn_fwd_prefill_ex(*prefill_args(), ctypes.cast(ctypes.byref(f), P)) == 1
    assert lib.attn_fwd_decode_ex(*decode_args(), ctypes.cast(ctypes.byref(f), P)) == 1
    qs = (ctypes.c_int64 * 3)(4096, 1024, 128)
    assert lib.attn_fwd_dense_ex(FAKE, FAKE, FAKE, FAKE, qs, qs, qs, qs, 2, 32, 16, 8, 2, 128,
                                 0.088, 1, 1, 0, None, None, None,
                                 ctypes.cast(ctypes.byref(f), P)) == 1


def test_valid_feature_flags_pass_validation(lib):
    """Valid flags on an empty problem: the call is a no-op that returns OK
    without touching a GPU."""
    import attention_forward_sdpa_gb300 as pkg
    pkg.load_library()
    f = pkg._Features(128, 0, 30.0, None, None)
    P = ctypes.POINTER(pkg._Features)
    assert lib.attn_fwd_prefill_ex(*prefill_args(num_seqs=0), ctypes.cast(ctypes.byref(f), P)) == 0
    assert lib.attn_fwd_prefill_ex(*prefill_args(num_seqs=0), None) == 0


def test_round_rejects_bad_arguments(lib):
    assert lib.attn_round_f32(FAKE, FAKE, -1, 1, 0, None) == 1
    assert lib.attn_round_f32(FAKE, FAKE, 10, 1, 3, None) == 1
    assert lib.attn_round_f32(None, FAKE, 10, 1, 0, None) == 1
    assert lib.attn_round_f32(ctypes.c_void_p(0x10001), FAKE, 10, 1, 0, None) == 1   # 2-byte out
    assert lib.attn_round_f32(FAKE, ctypes.c_void_p(0x10002), 10, 1, 0, None) == 1   # 4-byte in
    assert lib.attn_round_f32(FAKE, FAKE, 0, 1, 0, None) == 0


def test_binding_refuses_cpu_tensors(lib):
    import attention_forward_sdpa_gb300 as attn
    q = torch.zeros(4, 2, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 16, 2, 64, dtype=torch.bfloat16)
    bt = torch.zeros(1, 1, dtype=torch.int32)
    with pytest.raises(ValueError):
        attn.attn_fwd_prefill(torch.empty_like(q), q, k, k, bt, torch.tensor([0, 4], dtype=torch.int32),
                              torch.tensor([4], dtype=torch.int32), max_seqlen_q=4, max_seqlen_k=4,
                              scale=0.125, causal=True)
    with pytest.raises(TypeError):
        attn.prefill(q.float(), k, k, bt, torch.tensor([0, 4], dtype=torch.int32),
                     torch.tensor([4], dtype=torch.int32), max_seqlen_q=4, max_seqlen_k=4)


def fp8_feat(pkg, kv_fp8=1, k_scale=0.5, v_scale=2.0, ws=None, ws_bytes=0):
    return pkg._Features(-1, -1, 0.0, None, None, kv_fp8, k_scale, v_scale, ws, ws_bytes)


@pytest.mark.parametrize("kv_fp8,k_scale,v_scale", [
    (2, 1.0, 1.0), (-1, 1.0, 1.0),                 # flag outside {0, 1}
    (1, 0.0, 1.0), (1, -1.0, 1.0),                 # factors not positive
    (1, 1.0, float("nan")), (1, float("inf"), 1.0),
])
def test_fp8_fields_are_validated(lib, kv_fp8, k_scale, v_scale):
    import attention_forward_sdpa_gb300 as pkg
    pkg.load_library()
    P = ctypes.POINTER(pkg._Features)
    f = fp8_feat(pkg, kv_fp8, k_scale, v_scale, FAKE, 1 << 30)
    assert lib.attn_fwd_prefill_ex(*prefill_args(), ctypes.cast(ctypes.byref(f), P)) == 1
    assert lib.attn_fwd_decode_ex(*decode_args(), ctypes.cast(ctypes.byref(f), P)) == 1


def test_fp8_calls_need_their_workspace(lib):
    import attention_forward_sdpa_gb300 as pkg
    pkg.load_library()
    P = ctypes.POINTER(pkg._Features)
    need = lib.attn_fp8_prefill_workspace_size(2, 200, 2, 128, 64)
    for ws, nbytes in ((None, 0), (FAKE, need - 1), (ctypes.c_void_p(0x10010), need)):
        f = fp8_feat(pkg, ws=ws, ws_bytes=nbytes)   # missing, short, misaligned
        assert lib.attn_fwd_prefill_ex(*prefill_args(), ctypes.cast(ctypes.byref(f), P)) == 4
    # dense: batch 2, Sq 32, Sk 16, Hq 8, Hkv 2, d 128; its workspace is the
    # prefill one with one page of Sk rows per batch entry
    qs = (ctypes.c_int64 * 3)(4096, 1024, 128)
    kvs = (ctypes.c_int64 * 3)(16 * 2 * 128, 2 * 128, 128)
    need_d = lib.attn_fp8_prefill_workspace_size(2, 16, 2, 128, 16)
    for ws, nbytes in ((None, 0), (FAKE, need_d - 1)):
        f = fp8_feat(pkg, ws=ws, ws_bytes=nbytes)
        assert lib.attn_fwd_dense_ex(FAKE, FAKE, FAKE, FAKE, qs, kvs, kvs, qs, 2, 32, 16, 8, 2,
                                     128, 0.088, 1, 1, 0, None, None, None,
                                     ctypes.cast(ctypes.byref(f), P)) == 4
    # fp8 strides are in bytes and must be multiples of 16
    bad = (ctypes.c_int64 * 3)(16 * 2 * 128, 2 * 128 + 8, 128)
    f = fp8_feat(pkg, ws=FAKE, ws_bytes=need_d)
    assert lib.attn_fwd_dense_ex(FAKE, FAKE, FAKE, FAKE, qs, bad, kvs, qs, 2, 32, 16, 8, 2, 128,
                                 0.088, 1, 1, 0, None, None, None,
                                 ctypes.cast(ctypes.byref(f), P)) == 1


def test_fp8_prefill_workspace_size_is_arithmetic(lib):
    # 2 sequences x ceil(200 / 64) = 4 pages of 64 x 2 x 128 elements, two
    # 16-bit copies (K, V), then the 8-entry block table rounded up to 256 bytes
    assert lib.attn_fp8_prefill_workspace_size(2, 200, 2, 128, 64) == 2 * 8 * 16384 * 2 + 256
    assert lib.attn_fp8_prefill_workspace_size(0, 200, 2, 128, 64) == 0
    assert lib.attn_fp8_prefill_workspace_size(1, 0, 1, 64, 16) == 2 * 1024 * 2 + 256


def test_header_is_plain_c_and_links(lib, tmp_path):
    """A C99 program (no C++) includes include/attn_fwd.h without a warning
    under -Wall -Wextra -pedantic, links against the shared library and calls
    two entry points that need no GPU."""
    import subprocess
    import attention_forward_sdpa_gb300 as pkg
    src = tmp_path / "use_header.c"
    src.write_text('#include "attn_fwd.h"\n#include <stdio.h>\n'
                   "int main(void) {\n"
                   '  printf("%d|%s\\n", (int)attn_abi_version(),\n'
                   "         attn_status_string(ATTN_ERR_BAD_BLOCK_TABLE));\n"
                   "  return attn_decode_workspace_size(2, 4, 128, 1) == 256 ? 0 : 1;\n"
                   "}\n")
    exe = tmp_path / "use_header"
    libdir = os.path.dirname(pkg.library_path())
    cc = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                         f"-I{HEADER_DIR}", str(src), f"-L{libdir}", "-lattn_fwd_sm103",
                         f"-Wl,-rpath,{libdir}", "-o", str(exe)], capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stderr
    assert run.stdout.strip() == "2|block table entry out of range"

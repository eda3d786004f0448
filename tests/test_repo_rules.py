"""Static checks of the separation between the product and its test
infrastructure (CPU):

  - the package and the C boundary never reference the oracle (only the
    tests, the smoke check and the bench's CPU legs may run it), and the
    oracle never references the package or the CUDA sources: the two share
    no code;
  - the seeded input module holds no attention arithmetic of its own (it
    imports neither side);
  - no committed file points into the untracked working folder.
"""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "attention_forward_sdpa_gb300")
SKIP_DIRS = {".git", "_work", "gpurun_out", "__pycache__", "_build", "baseline", ".pytest_cache"}


def files_under(top, exts):
    for dirpath, dirnames, filenames in os.walk(top):
        dirnames[:] = [d for d in dirnames if d not in SKIP_DIRS]
        for f in filenames:
            if f.endswith(exts):
                yield os.path.join(dirpath, f)


def read(path):
    with open(path, encoding="utf-8", errors="replace") as f:
        return f.read()


def test_product_never_references_the_oracle():
    for path in files_under(PKG, (".py", ".cu", ".cuh", ".h", ".cpp")):
        text = read(path)
        assert not re.search(r"^\s*(from|import)\s+oracle\b", text, flags=re.M), path
        assert "sdpa_oracle" not in text, path
    for path in files_under(os.path.join(ROOT, "include"), (".h",)):
        assert "oracle" not in read(path).lower(), path


def test_oracle_never_references_the_product():
    for path in files_under(os.path.join(ROOT, "oracle"), (".py", ".c", ".h")):
        text = read(path)
        assert "attention_forward_sdpa_gb300" not in text, path
        assert "attn_fwd.h" not in text and "csrc" not in text, path
        assert not re.search(r"^\s*(from|import)\s+attn_inputs\b", text, flags=re.M), path


def test_input_generator_imports_neither_side():
    text = read(os.path.join(ROOT, "attn_inputs.py"))
    assert not re.search(r"^\s*(from|import)\s+(oracle|attention_forward_sdpa_gb300)\b", text,
                         flags=re.M)


def test_nothing_committed_points_into_the_working_folder():
    pattern = re.compile(r"(^|[\s'\"/(])_work/")
    for path in files_under(ROOT, (".py", ".cu", ".cuh", ".h", ".c", ".md", ".txt", ".json")):
        assert not pattern.search(read(path)), os.path.relpath(path, ROOT)


CSRC = os.path.join(PKG, "csrc")


def test_every_barrier_wait_in_the_kernels_is_bounded():
    """Every spin on an mbarrier gives up after a time limit (the kernels then
    record a timeout in the status word and leave), and no device code traps
    or asserts: a stalled pipeline cannot hang the GPU."""
    ptx = read(os.path.join(CSRC, "sm103_ptx.cuh"))
    assert ptx.count("mbarrier.try_wait") == 1          # only inside mbar_test
    wait = ptx[ptx.index("bool mbar_wait("):]
    wait = wait[:wait.index("\n}\n")]
    assert "global_timer_ns() - t0 > limit_ns" in wait and "*abort" in wait
    for path in files_under(CSRC, (".cu", ".cuh")):
        text = read(path)
        if not path.endswith("sm103_ptx.cuh"):
            assert "mbarrier.try_wait" not in text and "mbarrier.test_wait" not in text, path
        loops = list(re.finditer(r"while \(!mbar_test\([^)]*\)\) \{", text))
        if not path.endswith("sm103_ptx.cuh"):
            # a raw barrier probe appears only as the head of a bounded loop
            assert len(loops) == text.count("mbar_test("), path
        for m in loops:
            body = text[m.end():text.index("}", m.end())]
            assert "global_timer_ns() - t0 >" in body, (path, text[m.start():m.end()])
        code = re.sub(r"//[^\n]*|/\*.*?\*/", "", text, flags=re.S)
        assert "__trap" not in code and "brkpt" not in code, path
        assert not re.search(r"(?<!static_)assert\s*\(", code), path

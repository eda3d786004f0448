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

"""Host-side logic of bench.py (CPU only): the code fingerprint that decides
whether the recorded streaming-pass traffic still describes the kernels."""
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _topk_source():
    with open(os.path.join(ROOT, "gradient_compression_gb300", "csrc", "gc_topk.cu")) as fh:
        return fh.read()


def test_code_text_ignores_comments_and_blank_lines():
    src = _topk_source()
    edited = ("// a new leading comment\n\n" + src.replace("constexpr int FTHREADS = 512;",
                                                         "constexpr int FTHREADS = 512;  // noted\n\n   ")
              + "\n/* a block\n   comment */\n")
    assert edited != src
    assert bench.code_text(edited) == bench.code_text(src)


def test_code_text_sees_code_changes():
    src = _topk_source()
    changed = src.replace("constexpr int FTHREADS = 512;", "constexpr int FTHREADS = 256;")
    assert changed != src
    assert bench.code_text(changed) != bench.code_text(src)


def test_code_text_strips_both_comment_forms():
    assert bench.code_text("int a; // x\n/* y\n z */int b;\n\n  \nint c;   \n") == "int a;\nint b;\nint c;"

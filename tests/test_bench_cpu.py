"""Host-side pieces of bench.py that need no GPU."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_source_code_only_drops_comments_and_whitespace():
    text = "int a = 1; // one\n/* block\n comment */ int  b =\n 2;\n"
    assert bench.source_code_only(text) == "inta=1;intb=2;"
    # a comment-only change keeps the hash, a code change does not
    base = {"f": "x = 1; // note"}
    same = {"f": "x  =  1;   /* another note */"}
    other = {"f": "x = 2; // note"}
    saved = bench.KERNEL_SOURCES
    try:
        bench.KERNEL_SOURCES = ["f"]
        h0 = bench.kernel_source_hash(lambda f: base[f])
        assert bench.kernel_source_hash(lambda f: same[f]) == h0
        assert bench.kernel_source_hash(lambda f: other[f]) != h0
    finally:
        bench.KERNEL_SOURCES = saved


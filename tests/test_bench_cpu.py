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



def test_layer_row_fractions():
    import workloads as wl
    call = wl.ladder().calls[1]  # 128 -> 128 at [17, 256, 256]
    pk = {"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0, "hbm_gbs": 6400.0}
    ms = call.flops / 1000e12 * 1e3  # 1000 TFLOP/s
    row = bench.layer_row(call, ms, pk, 1, wl.NDHWC, "ladder")
    assert abs(row["tflops"] - 1000.0) < 0.2
    assert row["frac_bf16"] == 0.5 and row["frac_bf16_sustained"] == 0.625
    gbs = call.bytes() / (ms * 1e-3) / 1e9
    assert abs(row["frac_hbm"] - gbs / 6400.0) < 1e-3
    assert abs(row["frac_hbm_nominal"] - gbs / 8000.0) < 1e-3

"""Host-side pieces of bench.py that need no GPU."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_fingerprint_ignores_comments_and_whitespace(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("int f(int x) {\n    return x + 1;   // add one\n}\n")
    b = tmp_path / "b.cu"
    b.write_text("/* a comment\n   over lines */\nint f(int x) { return x + 1; }\n// trailing\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) {\n    return x + 2;   // add one\n}\n")
    assert bench.code_fingerprint(str(a)) == bench.code_fingerprint(str(b))
    assert bench.code_fingerprint(str(a)) != bench.code_fingerprint(str(c))


def test_measured_traffic_matches_the_committed_kernel():
    # the counters recorded in bench.py came from the GEMM code as committed
    bytes_, source = bench.measured_traffic("gemm_fp8_block", 585209651)
    assert bytes_ is not None, source
    assert 0 < bytes_ < 2 * 585209651
    assert bench.measured_traffic("no_such_kernel", 1) == (None, None)

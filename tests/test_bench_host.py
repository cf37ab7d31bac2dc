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


def test_host_cpu_reads_x86_and_arm_cpuinfo(tmp_path):
    x86 = tmp_path / "x86"
    x86.write_text("processor\t: 0\nmodel name\t: Some CPU @ 2.0GHz\n\nprocessor\t: 1\nmodel name\t: Some CPU @ 2.0GHz\n")
    assert bench.host_cpu(str(x86))["cpu_model"] == "Some CPU @ 2.0GHz"
    arm = tmp_path / "arm"
    arm.write_text("processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\nCPU part\t: 0xd4f\n")
    got = bench.host_cpu(str(arm))
    assert "implementer 0x41 part 0xd4f" in got["cpu_model"] and got["cpu_count"] >= 1
    assert bench.host_cpu(str(tmp_path / "missing"))["cpu_model"]

"""Host logic of bench.py on the CPU: which forward kernel a layer runs (as the library
dispatches it), the roofline and kernel-map byte counts, the traffic figure taken from a
committed ncu summary only while the kernel source matches it, and the per-step spread."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("I,O,kernel", [(64, 64, "fwd_tm"), (16, 48, "fwd_tm"), (32, 32, "fwd_tm"),
                                        (128, 128, "fwd_tc_tg"), (64, 128, "fwd_tc_tg"),
                                        (192, 80, "fwd_tc_tg"), (256, 256, "fwd_tc_tg"),
                                        (128, 256, "fwd_tc_tg"), (96, 96, "fwd_tc"),
                                        (72, 136, "fwd_tc"), (24, 40, "fwd_tc")])
def test_forward_kernel_follows_the_dispatch(I, O, kernel):
    name, src = bench.forward_kernel(I, O)
    assert name == kernel
    assert os.path.exists(src)


def test_kmap_bytes_closed_forms():
    N = 2_923_905
    assert bench.kmap_algorithmic_bytes(N, False, 0) == 172 * N
    assert bench.kmap_algorithmic_bytes(N, True, 1) == 176 * N
    # windows of 2^18: the last window is number 11, four bits above the 27-bit mask ->
    # 31-bit grouping keys, ceil(31 / 8) = 4 passes
    w = 1 << 18
    passes = (27 + ((N - 1) // w).bit_length() + 7) // 8
    assert passes == 4
    assert bench.kmap_algorithmic_bytes(N, True, w) == (172 + 12 + 24 * passes + 20 + 216) * N


def test_roofline_figures_are_consistent():
    N, P, I, O = 2_923_905, 31_178_577, 64, 64
    peaks = {"hbm_gbs": 6500.0, "bf16_tflops": 1700.0}
    r = bench.roofline(N, P, I, O, 840e-6, peaks, "measured", "shells16_1024_morton")
    gathered = P * I * 2 + N * O * 2 + 108 * N + 27 * I * O * 2
    assert r["algorithmic_bytes"] == gathered
    assert r["achieved"] == pytest.approx(gathered / 840e-6 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6500.0)
    assert r["tensor_tflops"] == pytest.approx(2.0 * P * I * O / 840e-6 / 1e12)
    assert r["kernel"] == "fwd_tm" and r["bound"] == "hbm"
    # fp32 runs the CUDA-core kernel and counts four bytes per element
    r32 = bench.roofline(N, P, I, O, 840e-6, peaks, "measured", "x", e=4)
    assert r32["kernel"] == "fwd_simt"
    assert r32["algorithmic_bytes"] == P * I * 4 + N * O * 4 + 108 * N + 27 * I * O * 4
    # the residual read of the fused epilogue adds N*O elements
    rr = bench.roofline(N, P, I, O, 840e-6, peaks, "measured", "x", residual=True)
    assert rr["algorithmic_bytes"] == gathered + N * O * 2


def test_traffic_only_from_a_summary_of_the_current_source():
    prof = os.path.join(ROOT, "profiles", "fwd_tm_shells16_1024_morton.md")
    src = os.path.join(bench.CSRC, "forward_tm.cu")
    t, how = bench.recorded_traffic("fwd_tm", src, "shells16_1024_morton")
    import hashlib
    import re
    text = open(prof).read()
    same = re.search(r"source_sha256:\s*([0-9a-f]{64})", text).group(1) == \
        hashlib.sha256(open(src, "rb").read()).hexdigest()
    if same:
        assert t == float(re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text).group(1))
        assert "profiles" in how
    else:
        assert t is None and how == "kernel changed since the ncu capture"
    # another source file than the one captured: never a traffic figure
    t2, how2 = bench.recorded_traffic("fwd_tm", os.path.join(bench.CSRC, "kmap.cu"),
                                      "shells16_1024_morton")
    assert t2 is None and how2 == "kernel changed since the ncu capture"
    assert bench.recorded_traffic("fwd_tm", src, "no_such_workload") == (None, "no ncu summary")


def test_spread_reports_the_slowest_step():
    s = bench.spread([3.0, 1.0, 7.0, 2.0])
    assert s["min"] == 1.0 and s["max"] == 7.0 and s["max_at_step"] == 2
    assert s["median"] == 2.5 and s["mean"] == pytest.approx(13.0 / 4)

"""bench.py's contract helpers, without a GPU: the credited FLOPs per step
(4 B H N^2 d forward, 2.5x that backward, halved under the causal mask, i.e.
1.0995e12 / 2.749e12 at B=2 H=16 N=8192 d=128 and 2.199e12 / 5.498e12 for the
causal B=1 H=8 N=32768 d=128 case), the comment-blind source hash, and the
rule that a committed DRAM-traffic line is used only while the kernel's
sources still hash to the value recorded with it."""
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_credited_flops():
    f, b = bench.flops_per_step(2, 16, 8192, 128, False)
    assert f == pytest.approx(1.0995e12, rel=1e-4) and b == pytest.approx(2.749e12, rel=1e-4)
    f, b = bench.flops_per_step(1, 8, 32768, 128, True)
    assert f == pytest.approx(2.199e12, rel=1e-4) and b == pytest.approx(5.498e12, rel=1e-4)


def test_code_only_ignores_comments_and_layout():
    a = "int x = 1; // one\n/* block\ncomment */ int y =  2;\n"
    b = "int x = 1;\nint y = 2;"
    assert bench.code_only(a) == bench.code_only(b) == "int x = 1; int y = 2;"
    assert bench.code_only("int x = 1;") != bench.code_only("int x = 2;")


def test_traffic_lines_follow_the_source_hash(monkeypatch):
    lines = [ln for ln in open(os.path.join(ROOT, "profiles", "dram_traffic.txt")).read().splitlines()
             if ln.strip() and not ln.startswith("#")]
    assert lines
    for ln in lines:
        kv = dict(tok.split("=", 1) for tok in ln.split())
        assert int(kv["dram_bytes_per_launch"]) > 0
        assert kv["kernel"] in bench.KERNEL_SOURCES
    kv = dict(tok.split("=", 1) for tok in lines[0].split())
    # the recorded hash: the line is used; any other hash: it is not
    monkeypatch.setattr(bench, "sources_sha", lambda kernel: kv["sources_sha"])
    assert bench.traffic_from_profiles(kv["kernel"], kv["config"]) == float(kv["dram_bytes_per_launch"])
    monkeypatch.setattr(bench, "sources_sha", lambda kernel: "0" * 16)
    assert bench.traffic_from_profiles(kv["kernel"], kv["config"]) is None
    assert bench.traffic_from_profiles(kv["kernel"], "no_such_config") is None


def test_source_hash_covers_every_listed_file():
    for kernel, files in bench.KERNEL_SOURCES.items():
        for name in files:
            assert os.path.exists(os.path.join(ROOT, "io_aware_exact_12_gb300", "csrc", name)), name
        assert len(bench.sources_sha(kernel)) == 16


def test_peaks_have_the_roofline_denominators():
    peaks, source = bench.load_peaks()
    assert source in ("measured", "fallback")
    for key in ("bf16_tflops", "hbm_gbs"):
        assert float(peaks.get(key, bench.FALLBACK_PEAKS[key])) > 0

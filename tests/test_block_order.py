"""The causal kernels visit (block, head) pairs in a grouped heaviest-first
order computed on the device from the linear block index.  This builds the
same header function for the host (tests/block_order_check.cpp) and checks
that it is a bijection onto every (rank, head) pair for many grid shapes and
head-group sizes, with ranks non-decreasing within a group."""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_grouped_rank_order_is_a_bijection(tmp_path):
    exe = str(tmp_path / "block_order_check")
    cmd = ["g++", "-std=c++17", "-O1", "-Wall", "-I", os.path.join(ROOT, "io_aware_exact_12_gb300", "csrc"),
           os.path.join(ROOT, "tests", "block_order_check.cpp"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok")

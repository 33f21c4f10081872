"""The kernels' block-order helpers (block_order.h), built for the host by
tests/block_order_check.cpp: the causal kernels' grouped heaviest-first order
is a bijection onto every (rank, head) pair with ranks non-decreasing within a
group, and the backward's split of its last partial wave covers every item
(the split ones by both halves) for many grid and SM counts."""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_block_order_helpers(tmp_path):
    exe = str(tmp_path / "block_order_check")
    cmd = ["g++", "-std=c++17", "-O1", "-Wall", "-I", os.path.join(ROOT, "io_aware_exact_12_gb300", "csrc"),
           os.path.join(ROOT, "tests", "block_order_check.cpp"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok")

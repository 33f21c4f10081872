"""A plain-C program (tests/c_abi_example.c) built against include/attn.h and
libattn.so: it compiles and links without a GPU; with one it runs and checks
O = c for rows of V all equal to c, and zero gradients for dO = 0."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi_example.c")


def _cuda_dirs():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    inc = os.path.join(home, "include")
    libs = [p for p in (os.path.join(home, "lib64"), os.path.join(home, "lib"),
                        os.path.join(home, "targets", "sbsa-linux", "lib"),
                        os.path.join(home, "targets", "x86_64-linux", "lib"))
            if os.path.exists(os.path.join(p, "libcudart.so"))]
    return inc, libs


def _build(tmp_path):
    from io_aware_exact_12_gb300 import build as b
    lib = b.build()
    pkg = os.path.dirname(lib)
    inc, libs = _cuda_dirs()
    if not os.path.exists(os.path.join(inc, "cuda_runtime.h")) or not libs:
        pytest.skip("CUDA runtime headers or library not found")
    exe = str(tmp_path / "c_abi_example")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-I", os.path.join(ROOT, "include"), "-I", inc, SRC, "-o", exe,
           "-L", pkg, "-lattn", "-L", libs[0], "-lcudart", "-lm", "-Wl,-rpath," + pkg + ":" + libs[0]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_program_compiles_and_links(tmp_path):
    _build(tmp_path)


@pytest.mark.gpu
def test_c_program_runs_on_the_gpu(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok")

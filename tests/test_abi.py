"""C-ABI checks that need no GPU: the library builds and loads, exports every
function the headers under include/ declare (the attention ABI attn.h and the
diagnostics attn_diag.h), and rejects bad arguments synchronously (before
any CUDA call, so nothing is launched)."""
import ctypes
import os
import re

import pytest

from io_aware_exact_12_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))


@pytest.fixture(scope="module")
def L():
    path = build_mod.build()
    import io_aware_exact_12_gb300 as pkg
    return pkg.lib()


def declared_functions(headers=None):
    names = set()
    for h in headers or HEADERS:
        text = open(h, encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(attn_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions([os.path.join(ROOT, "include", "attn.h")])
    for required in ("attn_fwd", "attn_bwd", "attn_fwd_f16", "attn_bwd_f16", "attn_sync_status",
                     "attn_status_string"):
        assert required in names
    # the measurement aid and the failure-path self-test are not attention
    assert "attn_probe_ex2" not in names and "attn_debug_wait_timeout" not in names
    diag = declared_functions([os.path.join(ROOT, "include", "attn_diag.h")])
    assert diag == ["attn_debug_wait_timeout", "attn_probe_ex2"]


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings(L):
    for code in range(0, 7):
        s = L.attn_status_string(code)
        assert s and s != b"unknown status"
    assert L.attn_status_string(99) == b"unknown status"


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below fails validation first


def _fwd(L, q=FAKE, k=FAKE + 0x100000, v=FAKE + 0x200000, o=FAKE + 0x300000, lse=FAKE + 0x400000,
         B=1, H=1, N=16, d=64, scale=0.125, causal=0):
    return L.attn_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, None)


def test_fwd_rejects_bad_arguments(L):
    assert _fwd(L, q=None) == 1
    assert _fwd(L, lse=None) == 1
    assert _fwd(L, B=0) == 1
    assert _fwd(L, H=-1) == 1
    assert _fwd(L, N=0) == 1
    assert _fwd(L, scale=float("nan")) == 1
    assert _fwd(L, scale=float("inf")) == 1
    assert _fwd(L, d=48) == 2
    assert _fwd(L, d=256) == 2
    assert _fwd(L, B=300, H=300) == 2          # B*H beyond the grid limit
    assert _fwd(L, q=FAKE + 8) == 1            # misaligned
    assert _fwd(L, o=FAKE) == 1                # output aliases an input
    assert L.attn_fwd_f16(None, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 64, 0.125, 0, None) == 1


def test_bwd_rejects_bad_arguments(L):
    base = [FAKE + i * 0x100000 for i in range(9)]

    def bwd(**kw):
        a = list(base)
        names = ["q", "k", "v", "o", "do", "lse", "dq", "dk", "dv"]
        for n, val in kw.items():
            if n in names:
                a[names.index(n)] = val
        B, H, N, d = kw.get("B", 1), kw.get("H", 2), kw.get("N", 100), kw.get("d", 128)
        return L.attn_bwd(*a, B, H, N, d, kw.get("scale", 0.1), 1, None)

    assert bwd(dq=None) == 1
    assert bwd(N=0) == 1
    assert bwd(d=96) == 2
    assert bwd(dk=base[0]) == 1                # gradient aliases q
    assert bwd(dv=base[6]) == 1                # dv aliases dq
    assert bwd(lse=FAKE + 0x500002) == 1       # lse not 4-byte aligned


def test_ex2_probe_rejects_bad_arguments(L):
    assert L.attn_probe_ex2(None, 1, 1, None) == 1
    assert L.attn_probe_ex2(FAKE, 0, 1, None) == 1
    assert L.attn_probe_ex2(FAKE, 65536, 1, None) == 1
    assert L.attn_probe_ex2(FAKE, 1, 0, None) == 1
    assert L.attn_probe_ex2(FAKE, 1, (1 << 20) + 1, None) == 1
    assert L.attn_probe_ex2(FAKE + 2, 1, 1, None) == 1  # not 4-byte aligned


def test_valid_arguments_without_gpu_report_an_error(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: a call with fake pointers would launch")
    rc = _fwd(L)
    assert rc in (3, 5)  # no CUDA device here: runtime error or wrong architecture, never a launch


def test_dropout_rejects_bad_probability(L):
    args = [FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000, FAKE + 0x400000, 1, 1, 16, 64, 0.125, 0]
    for p in (1.0, -0.1, float("nan"), 0.999):
        assert L.attn_fwd_dropout(*args, p, 1, 0, None) == 1
    bargs = [FAKE + i * 0x100000 for i in range(9)] + [1, 2, 100, 128, 0.1, 1]
    assert L.attn_bwd_dropout(*bargs, 1.5, 1, 0, None) == 1
    assert L.attn_bwd_dropout(*bargs[:9], 1, 2, 100, 96, 0.1, 1, 0.1, 1, 0, None) == 2


def test_blocksparse_backward_rejects_bad_arguments(L):
    a = [FAKE + i * 0x100000 for i in range(9)]
    assert L.attn_bwd_blocksparse(*a, None, 1, 1, 2, 256, 128, 0.1, 0, None) == 1       # no mask
    assert L.attn_bwd_blocksparse(*a, FAKE, 3, 1, 2, 256, 128, 0.1, 0, None) == 1       # mask_heads not 1 or H
    assert L.attn_bwd_blocksparse(*a, FAKE, 1, 1, 2, 262144 + 128, 128, 0.1, 0, None) == 2  # > 2048 tiles


def test_blocksparse_dropout_rejects_bad_arguments(L):
    fa = [FAKE + i * 0x100000 for i in range(5)]
    assert L.attn_fwd_blocksparse_dropout(*fa, None, 1, 1, 2, 256, 128, 0.1, 0, 0.1, 1, 0, None) == 1   # no mask
    assert L.attn_fwd_blocksparse_dropout(*fa, FAKE, 3, 1, 2, 256, 128, 0.1, 0, 0.1, 1, 0, None) == 1   # mask_heads
    assert L.attn_fwd_blocksparse_dropout(*fa, FAKE, 1, 1, 2, 256, 128, 0.1, 0, 1.0, 1, 0, None) == 1   # p_drop
    assert L.attn_fwd_blocksparse_dropout_f16(*fa, FAKE, 1, 1, 2, 256, 96, 0.1, 0, 0.1, 1, 0, None) == 2  # d
    a = [FAKE + i * 0x100000 for i in range(9)]
    assert L.attn_bwd_blocksparse_dropout(*a, None, 1, 1, 2, 256, 128, 0.1, 0, 0.1, 1, 0, None) == 1
    assert L.attn_bwd_blocksparse_dropout(*a, FAKE, 1, 1, 2, 256, 128, 0.1, 0, -0.5, 1, 0, None) == 1
    assert L.attn_bwd_blocksparse_dropout_f16(*a, FAKE, 1, 1, 2, 262144 + 128, 128, 0.1, 0, 0.1, 1, 0,
                                              None) == 2  # > 2048 tiles

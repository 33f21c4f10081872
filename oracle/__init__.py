"""Float64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this package.  The
CUDA library never imports, links or calls it, and it shares no code with
the CUDA library: the two meet only through the seeded inputs of
``io_aware_exact_12_gb300.synth`` (which holds none of the method's
arithmetic).

``attn_oracle.c`` is the plain definition (materialising S, P and O, and the
analytic backward); ``blockwise.py`` is an independent NumPy restatement of
the online-softmax recurrences used to cross-check it.  See those files for
the passages each function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c with gcc into oracle/liboracle.so (plain C, -O2)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_forward.argtypes = [P, P, P, P, P, P, I64, I64, I64, ctypes.c_double, ctypes.c_int, ctypes.c_int]
        lib.oracle_forward_masked.argtypes = [P, P, P, P, P, P, I64, I64, I64, ctypes.c_double, ctypes.c_int, P,
                                              I64, I64, ctypes.c_int]
        lib.oracle_backward_masked.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I64, ctypes.c_double,
                                               ctypes.c_int, P, I64, I64, ctypes.c_int]
        lib.oracle_backward.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I64, ctypes.c_double, ctypes.c_int,
                                        ctypes.c_int]
        lib.oracle_rows.argtypes = [P, P, P, P, I64, I64, I64, ctypes.c_double, ctypes.c_int, P, P, I64, P, P, P,
                                    ctypes.c_int]
        lib.oracle_cols.argtypes = [P, P, P, P, P, P, I64, I64, I64, ctypes.c_double, ctypes.c_int, P, P, I64, P,
                                    P, ctypes.c_int]
        D, U64, U32 = ctypes.c_double, ctypes.c_uint64, ctypes.c_uint32
        lib.oracle_philox4x32_10.argtypes = [P, P, P]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_dropout_keep.argtypes = [D, U64, U32, I64, I64, I64, P]
        lib.oracle_forward_dropout.argtypes = [P, P, P, P, P, P, I64, I64, I64, D, ctypes.c_int, D, U64, U32,
                                               ctypes.c_int]
        lib.oracle_backward_dropout.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I64, D, ctypes.c_int, D, U64,
                                                U32, ctypes.c_int]
        lib.oracle_rows_dropout.argtypes = [P, P, P, P, I64, I64, I64, D, ctypes.c_int, D, U64, U32, P, P, I64, P,
                                            P, P, ctypes.c_int]
        lib.oracle_cols_dropout.argtypes = [P, P, P, P, P, P, I64, I64, I64, D, ctypes.c_int, D, U64, U32, P, P,
                                            I64, P, P, ctypes.c_int]
        lib.oracle_forward_masked_dropout.argtypes = [P, P, P, P, P, P, I64, I64, I64, D, ctypes.c_int, P, I64,
                                                      I64, D, U64, U32, ctypes.c_int]
        lib.oracle_backward_masked_dropout.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I64, D, ctypes.c_int, P,
                                                       I64, I64, D, U64, U32, ctypes.c_int]
        for f in (lib.oracle_forward, lib.oracle_backward, lib.oracle_rows, lib.oracle_cols,
                  lib.oracle_forward_masked, lib.oracle_backward_masked, lib.oracle_dropout_keep,
                  lib.oracle_forward_dropout, lib.oracle_backward_dropout, lib.oracle_rows_dropout,
                  lib.oracle_cols_dropout, lib.oracle_forward_masked_dropout,
                  lib.oracle_backward_masked_dropout):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _shape(q):
    if q.ndim != 4:
        raise ValueError("expected [B, H, N, d] arrays")
    return q.shape


def _mask(block_mask, H, N, blk):
    if block_mask is None:
        return None, 0
    m = np.ascontiguousarray(np.asarray(block_mask), dtype=np.uint8)
    nb = (N + blk - 1) // blk
    if m.ndim != 3 or m.shape[1:] != (nb, nb) or m.shape[0] not in (1, H):
        raise ValueError("block_mask must be [H or 1, ceil(N/blk), ceil(N/blk)]")
    return m, m.shape[0]


def philox4x32_10(ctr, key):
    """Philox4x32-10 of a 4-word counter and 2-word key (uint32 each) -> 4 words."""
    c = (ctypes.c_uint32 * 4)(*[int(x) & 0xFFFFFFFF for x in ctr])
    kk = (ctypes.c_uint32 * 2)(*[int(x) & 0xFFFFFFFF for x in key])
    out = (ctypes.c_uint32 * 4)()
    _load().oracle_philox4x32_10(ctypes.cast(c, ctypes.c_void_p), ctypes.cast(kk, ctypes.c_void_p),
                                 ctypes.cast(out, ctypes.c_void_p))
    return [int(x) for x in out]


def dropout_keep(p, seed, offset, bh, n_rows, n_cols):
    """keep_ij in {0, 1} (uint8 [n_rows, n_cols]) of flattened head ``bh``."""
    out = np.empty((n_rows, n_cols), dtype=np.uint8)
    rc = _load().oracle_dropout_keep(float(p), int(seed), int(offset), int(bh), n_rows, n_cols, _ptr(out))
    if rc:
        raise RuntimeError("oracle_dropout_keep failed (%d)" % rc)
    return out


def _drop(dropout):
    """dropout = (p, seed, offset) or None."""
    if dropout is None:
        return None
    p, seed, offset = dropout
    return float(p), int(seed), int(offset)


def forward(q, k, v, scale, causal, want_p=False, threads=None, block_mask=None, blk=128, dropout=None):
    """O, LSE (and optionally P) of softmax(scale q k^T [+ causal mask]) v.

    q, k, v: [B, H, N, d] (any float dtype; upcast exactly to float64).
    block_mask: optional [H or 1, nb, nb] (nb = ceil(N/blk)); key j is hidden
    from query i unless block_mask[h][i // blk][j // blk] is nonzero.
    dropout: optional (p, seed, offset): inverted dropout on P (P returned
    by want_p is the softmax before dropout; LSE is undropped); with a
    block_mask too, the keep rule applies to the keys the mask leaves visible.
    Returns (o [B,H,N,d], lse [B,H,N]) or (o, lse, p [B,H,N,N]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = _shape(q)
    o = np.empty_like(q)
    lse = np.empty((B, H, N), dtype=np.float64)
    p = np.empty((B, H, N, N), dtype=np.float64) if want_p else None
    m, mh = _mask(block_mask, H, N, blk)
    dr = _drop(dropout)
    if dr is not None and m is not None:
        rc = _load().oracle_forward_masked_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(p), B * H,
                                                   N, d, float(scale), int(bool(causal)), _ptr(m), mh, blk, *dr,
                                                   threads or default_threads())
    elif dr is not None:
        rc = _load().oracle_forward_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(p), B * H, N, d,
                                            float(scale), int(bool(causal)), *dr, threads or default_threads())
    elif m is None:
        rc = _load().oracle_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(p), B * H, N, d,
                                    float(scale), int(bool(causal)), threads or default_threads())
    else:
        rc = _load().oracle_forward_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(p), B * H, N, d,
                                           float(scale), int(bool(causal)), _ptr(m), mh, blk,
                                           threads or default_threads())
    if rc:
        raise RuntimeError("oracle_forward failed (%d)" % rc)
    return (o, lse, p) if want_p else (o, lse)


def backward(q, k, v, o, do, scale, causal, threads=None, block_mask=None, blk=128, dropout=None):
    """dQ, dK, dV of L = <O, dO>; ``o`` is the oracle's own forward output
    (with the same ``dropout``, when given)."""
    q, k, v, o, do = (_f64(x) for x in (q, k, v, o, do))
    B, H, N, d = _shape(q)
    dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
    m, mh = _mask(block_mask, H, N, blk)
    dr = _drop(dropout)
    if dr is not None and m is not None:
        rc = _load().oracle_backward_masked_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(dq),
                                                    _ptr(dk), _ptr(dv), B * H, N, d, float(scale),
                                                    int(bool(causal)), _ptr(m), mh, blk, *dr,
                                                    threads or default_threads())
    elif dr is not None:
        rc = _load().oracle_backward_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(dq), _ptr(dk),
                                             _ptr(dv), B * H, N, d, float(scale), int(bool(causal)), *dr,
                                             threads or default_threads())
    elif m is None:
        rc = _load().oracle_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                                     B * H, N, d, float(scale), int(bool(causal)), threads or default_threads())
    else:
        rc = _load().oracle_backward_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(dq), _ptr(dk),
                                            _ptr(dv), B * H, N, d, float(scale), int(bool(causal)), _ptr(m), mh,
                                            blk, threads or default_threads())
    if rc:
        raise RuntimeError("oracle_backward failed (%d)" % rc)
    return dq, dk, dv


def rows(q, k, v, do, scale, causal, bh_idx, row_idx, threads=None, dropout=None):
    """O rows, LSE and dQ rows for selected (flattened head, query row) pairs.

    Returns (o [n, d], lse [n], dq [n, d] or None when ``do`` is None).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    do = None if do is None else _f64(do)
    B, H, N, d = _shape(q)
    bh = np.ascontiguousarray(bh_idx, dtype=np.int64)
    ri = np.ascontiguousarray(row_idx, dtype=np.int64)
    n = bh.shape[0]
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    dq = np.empty((n, d), dtype=np.float64) if do is not None else None
    dr = _drop(dropout)
    if dr is not None:
        rc = _load().oracle_rows_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B * H, N, d, float(scale),
                                         int(bool(causal)), *dr, _ptr(bh), _ptr(ri), n, _ptr(o), _ptr(lse), _ptr(dq),
                                         threads or default_threads())
    else:
        rc = _load().oracle_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B * H, N, d, float(scale), int(bool(causal)),
                                 _ptr(bh), _ptr(ri), n, _ptr(o), _ptr(lse), _ptr(dq), threads or default_threads())
    if rc:
        raise RuntimeError("oracle_rows failed (%d)" % rc)
    return o, lse, dq


def cols(q, k, v, do, lse_all, D_all, scale, causal, bh_idx, col_idx, threads=None, dropout=None):
    """dK, dV rows for selected (flattened head, key) pairs.

    lse_all, D_all: [B, H, N] per-row LSE and D_i = sum_k dO_ik O_ik of every row.
    """
    q, k, v, do = (_f64(x) for x in (q, k, v, do))
    lse_all, D_all = _f64(lse_all), _f64(D_all)
    B, H, N, d = _shape(q)
    bh = np.ascontiguousarray(bh_idx, dtype=np.int64)
    ci = np.ascontiguousarray(col_idx, dtype=np.int64)
    n = bh.shape[0]
    dk = np.empty((n, d), dtype=np.float64)
    dv = np.empty((n, d), dtype=np.float64)
    dr = _drop(dropout)
    if dr is not None:
        rc = _load().oracle_cols_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse_all), _ptr(D_all), B * H, N,
                                         d, float(scale), int(bool(causal)), *dr, _ptr(bh), _ptr(ci), n, _ptr(dk),
                                         _ptr(dv), threads or default_threads())
    else:
        rc = _load().oracle_cols(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse_all), _ptr(D_all), B * H, N, d,
                                 float(scale), int(bool(causal)), _ptr(bh), _ptr(ci), n, _ptr(dk), _ptr(dv),
                                 threads or default_threads())
    if rc:
        raise RuntimeError("oracle_cols failed (%d)" % rc)
    return dk, dv

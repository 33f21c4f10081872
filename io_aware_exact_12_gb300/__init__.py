"""GB300 (sm_103a) fused exact attention: Python binding of the C ABI in
``include/attn.h``.

This module only marshals arguments: it checks tensor shapes/dtypes, allocates
outputs with torch (device memory and streams are the only things torch is
used for), and calls the same-named C entry points of ``libattn.so`` through
ctypes.  Every step of the computation runs in the library's CUDA kernels.
There is no fallback: if the library is missing or fails to load, every call
raises.

Layout: q, k, v, o, do and the gradients are contiguous [B, H, N, d] tensors
(bf16 or fp16) on one CUDA device; lse is fp32 [B, H, N].
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

__all__ = ["attention", "attn_fwd", "attn_bwd", "attn_fwd_dropout", "attn_bwd_dropout", "attn_decode", "attn_fwd_fp8", "attn_fwd_blocksparse", "attn_bwd_blocksparse",
           "attn_fwd_blocksparse_dropout", "attn_bwd_blocksparse_dropout", "sync_status", "status_string", "last_launch_count", "lib",
           "AttnError", "LIB_PATH", "STATUS"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libattn.so")

STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_CUDA",
          4: "ATTN_ERR_TIMEOUT", 5: "ATTN_ERR_ARCH", 6: "ATTN_ERR_DEVICE_CHECK"}


class AttnError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__("%s failed: %s (%d)" % (fn, STATUS.get(code, "?"), code))
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libattn.so not built; run `python -m io_aware_exact_12_gb300.build` "
                              "(or __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, F, I, P]
        L.attn_fwd_f16.argtypes = L.attn_fwd.argtypes
        L.attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, F, I, P]
        L.attn_bwd_f16.argtypes = L.attn_bwd.argtypes
        for f in (L.attn_fwd, L.attn_fwd_f16, L.attn_bwd, L.attn_bwd_f16):
            f.restype = I
        U64, U32 = ctypes.c_ulonglong, ctypes.c_uint
        for f in (L.attn_fwd_dropout, L.attn_fwd_dropout_f16):
            f.argtypes = [P, P, P, P, P, I, I, I, I, F, I, F, U64, U32, P]
            f.restype = I
        for f in (L.attn_bwd_dropout, L.attn_bwd_dropout_f16):
            f.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, F, I, F, U64, U32, P]
            f.restype = I
        for f in (L.attn_fwd_blocksparse, L.attn_fwd_blocksparse_f16):
            f.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, I, P]
            f.restype = I
        for f in (L.attn_bwd_blocksparse, L.attn_bwd_blocksparse_f16):
            f.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, I, P]
            f.restype = I
        for f in (L.attn_fwd_blocksparse_dropout, L.attn_fwd_blocksparse_dropout_f16):
            f.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, I, F, U64, U32, P]
            f.restype = I
        for f in (L.attn_bwd_blocksparse_dropout, L.attn_bwd_blocksparse_dropout_f16):
            f.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, I, F, U64, U32, P]
            f.restype = I
        L.attn_fwd_fp8.argtypes = [P, P, P, F, F, F, P, P, I, I, I, I, F, I, P]
        L.attn_fwd_fp8.restype = I
        L.attn_decode.argtypes = [P, P, P, P, P, I, I, I, I, F, P]
        L.attn_decode.restype = I
        L.attn_sync_status.argtypes = [P]
        L.attn_sync_status.restype = I
        L.attn_status_string.argtypes = [I]
        L.attn_status_string.restype = ctypes.c_char_p
        L.attn_last_launch_count.argtypes = []
        L.attn_last_launch_count.restype = I
        L.attn_probe_ex2.argtypes = [P, I, I, P]
        L.attn_probe_ex2.restype = I
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().attn_status_string(int(code)).decode()


def last_launch_count() -> int:
    return lib().attn_last_launch_count()


EX2_PROBE_THREADS = 256
EX2_PROBE_CHAINS = 8


def probe_ex2(sink, blocks, iters, stream=None):
    """Enqueue the exponential-unit throughput probe (attn_probe_ex2) writing
    one float per thread into `sink` (a float32 CUDA tensor of at least
    blocks * 256 elements).  Returns the number of exponentials it computes."""
    if not isinstance(sink, torch.Tensor) or not sink.is_cuda or sink.dtype != torch.float32:
        raise TypeError("sink must be a float32 CUDA tensor")
    if not sink.is_contiguous() or sink.numel() < blocks * EX2_PROBE_THREADS:
        raise ValueError("sink must be contiguous with at least blocks * 256 elements")
    with _on_device(sink):
        rc = lib().attn_probe_ex2(sink.data_ptr(), int(blocks), int(iters), _stream_handle(stream))
    if rc != 0:
        raise RuntimeError("attn_probe_ex2: %s" % status_string(rc))
    return blocks * EX2_PROBE_THREADS * iters * EX2_PROBE_CHAINS


class _Nothing:
    def __enter__(self):
        return None

    def __exit__(self, *exc):
        return False


_NOTHING = _Nothing()


def _on_device(t):
    """The C ABI works on the current device: switch to t's device only when
    it is not already current (entering torch.cuda.device costs several us)."""
    idx = t.device.index
    if idx is None or idx == torch.cuda.current_device():
        return _NOTHING
    return torch.cuda.device(t.device)


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(name, t, like=None, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous [B, H, N, d]" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s" % (name, dtype))
    if like is not None and (t.shape != like.shape or t.device != like.device):
        raise ValueError("%s must match q's shape/device" % name)


def _dims(q):
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("q must be bf16 or fp16")
    return tuple(int(x) for x in q.shape)


def attn_fwd(q, k, v, scale=None, causal=False, o=None, lse=None, stream=None):
    """O, LSE = exact softmax(scale q k^T [+ causal]) v.  Returns (o, lse)."""
    B, H, N, d = _dims(q)
    _check("q", q)
    _check("k", k, q, q.dtype)
    _check("v", v, q, q.dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check("o", o, q, q.dtype)
    _check("lse", lse, None, torch.float32)
    fn = lib().attn_fwd if q.dtype == torch.bfloat16 else lib().attn_fwd_f16
    with _on_device(q):
        rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                float(scale), int(bool(causal)), _stream_handle(stream))
    if rc:
        raise AttnError("attn_fwd", rc)
    return o, lse


def attn_bwd(q, k, v, o, do, lse, scale=None, causal=False, dq=None, dk=None, dv=None, stream=None):
    """dQ, dK, dV of L = <O, dO> by recomputation from LSE.  Returns (dq, dk, dv)."""
    B, H, N, d = _dims(q)
    _check("q", q)
    for name, t in (("k", k), ("v", v), ("o", o), ("do", do)):
        _check(name, t, q, q.dtype)
    _check("lse", lse, None, torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check(name, t, q, q.dtype)
    fn = lib().attn_bwd if q.dtype == torch.bfloat16 else lib().attn_bwd_f16
    with _on_device(q):
        rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, float(scale), int(bool(causal)),
                _stream_handle(stream))
    if rc:
        raise AttnError("attn_bwd", rc)
    return dq, dk, dv


def attn_fwd_dropout(q, k, v, p_drop, seed, offset=0, scale=None, causal=False, o=None, lse=None, stream=None):
    """attn_fwd with inverted dropout of probability ``p_drop`` on P, the keep
    decisions drawn in the kernel from Philox4x32-10 keyed by ``seed`` (64-bit)
    with ``offset`` (32-bit) as the fourth counter word.  bf16 or fp16.
    Returns (o, lse); lse is that of the undropped softmax."""
    B, H, N, d = _dims(q)
    _check("q", q)
    _check("k", k, q, q.dtype)
    _check("v", v, q, q.dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q) if o is None else o
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check("o", o, q, q.dtype)
    _check("lse", lse, None, torch.float32)
    with _on_device(q):
        fn = lib().attn_fwd_dropout if q.dtype == torch.bfloat16 else lib().attn_fwd_dropout_f16
        rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H,
                N, d, float(scale), int(bool(causal)), float(p_drop),
                int(seed) & 0xFFFFFFFFFFFFFFFF, int(offset) & 0xFFFFFFFF,
                _stream_handle(stream))
    if rc:
        raise AttnError("attn_fwd_dropout", rc)
    return o, lse


def attn_bwd_dropout(q, k, v, o, do, lse, p_drop, seed, offset=0, scale=None, causal=False, dq=None, dk=None,
                     dv=None, stream=None):
    """Gradients of attn_fwd_dropout's output (same p_drop, seed, offset): the
    keep decisions are drawn again, not stored.  Returns (dq, dk, dv)."""
    B, H, N, d = _dims(q)
    _check("q", q)
    for name, t in (("k", k), ("v", v), ("o", o), ("do", do)):
        _check(name, t, q, q.dtype)
    _check("lse", lse, None, torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check(name, t, q, q.dtype)
    with _on_device(q):
        fn = lib().attn_bwd_dropout if q.dtype == torch.bfloat16 else lib().attn_bwd_dropout_f16
        rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                float(scale), int(bool(causal)), float(p_drop),
                int(seed) & 0xFFFFFFFFFFFFFFFF, int(offset) & 0xFFFFFFFF,
                _stream_handle(stream))
    if rc:
        raise AttnError("attn_bwd_dropout", rc)
    return dq, dk, dv


def attn_decode(q, k, v, scale=None, o=None, lse=None, stream=None):
    """One decode step: q [B, H, d] (or [B, H, 1, d]) against the cache k, v
    [B, H, L, d], bf16; every key visible.  Returns (o [B, H, d], lse [B, H])."""
    if q.dim() == 4:
        if q.shape[2] != 1:
            raise ValueError("decode takes one query token per (batch, head)")
        q = q.reshape(q.shape[0], q.shape[1], q.shape[3])
    if q.dim() != 3 or k.dim() != 4:
        raise ValueError("q must be [B, H, d] and k, v [B, H, L, d]")
    B, H, d = (int(x) for x in q.shape)
    Lk = int(k.shape[2])
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(name, t, None, torch.bfloat16)
    if tuple(k.shape) != (B, H, Lk, d) or tuple(v.shape) != (B, H, Lk, d):
        raise ValueError("k and v must be [B, H, L, d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device) if lse is None else lse
    _check("o", o, q, torch.bfloat16)
    _check("lse", lse, None, torch.float32)
    with _on_device(q):
        rc = lib().attn_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Lk,
                               d, float(scale), _stream_handle(stream))
    if rc:
        raise AttnError("attn_decode", rc)
    return o, lse


def _check_block_mask(block_mask, H, N):
    nb = (N + 127) // 128
    if (not isinstance(block_mask, torch.Tensor) or not block_mask.is_cuda or block_mask.dtype != torch.uint8
            or not block_mask.is_contiguous() or block_mask.dim() != 3
            or tuple(block_mask.shape[1:]) != (nb, nb) or block_mask.shape[0] not in (1, H)):
        raise ValueError("block_mask must be a contiguous uint8 CUDA tensor [H or 1, %d, %d]" % (nb, nb))


def _fwd_blocksparse(name, q, k, v, block_mask, scale, causal, o, lse, stream, drop=None):
    B, H, N, d = _dims(q)
    _check("q", q)
    _check("k", k, q, q.dtype)
    _check("v", v, q, q.dtype)
    _check_block_mask(block_mask, H, N)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check("o", o, q, q.dtype)
    _check("lse", lse, None, torch.float32)
    args = [q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
            block_mask.data_ptr(), int(block_mask.shape[0]), B, H, N, d, float(scale), int(bool(causal))]
    if drop is not None:
        p_drop, seed, offset = drop
        args += [float(p_drop), int(seed) & 0xFFFFFFFFFFFFFFFF, int(offset) & 0xFFFFFFFF]
    with _on_device(q):
        fn = getattr(lib(), name if q.dtype == torch.bfloat16 else name + "_f16")
        rc = fn(*args, _stream_handle(stream))
    if rc:
        raise AttnError(name, rc)
    return o, lse


def _bwd_blocksparse(name, q, k, v, o, do, lse, block_mask, scale, causal, dq, dk, dv, stream, drop=None):
    B, H, N, d = _dims(q)
    _check("q", q)
    for n, t in (("k", k), ("v", v), ("o", o), ("do", do)):
        _check(n, t, q, q.dtype)
    _check("lse", lse, None, torch.float32)
    _check_block_mask(block_mask, H, N)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check(n, t, q, q.dtype)
    args = [q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), block_mask.data_ptr(), int(block_mask.shape[0]),
            B, H, N, d, float(scale), int(bool(causal))]
    if drop is not None:
        p_drop, seed, offset = drop
        args += [float(p_drop), int(seed) & 0xFFFFFFFFFFFFFFFF, int(offset) & 0xFFFFFFFF]
    with _on_device(q):
        fn = getattr(lib(), name if q.dtype == torch.bfloat16 else name + "_f16")
        rc = fn(*args, _stream_handle(stream))
    if rc:
        raise AttnError(name, rc)
    return dq, dk, dv


def attn_fwd_blocksparse(q, k, v, block_mask, scale=None, causal=False, o=None, lse=None, stream=None):
    """Forward restricted by a block mask: block_mask is a uint8 CUDA tensor
    [H or 1, ceil(N/128), ceil(N/128)]; key j is visible to query i iff
    block_mask[h][i // 128][j // 128] != 0 (and j <= i if causal).
    bf16 or fp16.  Returns (o, lse); rows that see no key get O = 0,
    LSE = -inf."""
    return _fwd_blocksparse("attn_fwd_blocksparse", q, k, v, block_mask, scale, causal, o, lse, stream)


def attn_bwd_blocksparse(q, k, v, o, do, lse, block_mask, scale=None, causal=False, dq=None, dk=None, dv=None,
                         stream=None):
    """Gradients of attn_fwd_blocksparse's output for the same block_mask and
    causal flag.  Returns (dq, dk, dv)."""
    return _bwd_blocksparse("attn_bwd_blocksparse", q, k, v, o, do, lse, block_mask, scale, causal, dq, dk, dv,
                            stream)


def attn_fwd_blocksparse_dropout(q, k, v, block_mask, p_drop, seed, offset=0, scale=None, causal=False, o=None,
                                 lse=None, stream=None):
    """attn_fwd_blocksparse with the dropout of attn_fwd_dropout on the keys
    the mask leaves visible (the keep decisions do not depend on the mask).
    Returns (o, lse); lse is that of the undropped softmax."""
    return _fwd_blocksparse("attn_fwd_blocksparse_dropout", q, k, v, block_mask, scale, causal, o, lse, stream,
                            (p_drop, seed, offset))


def attn_bwd_blocksparse_dropout(q, k, v, o, do, lse, block_mask, p_drop, seed, offset=0, scale=None,
                                 causal=False, dq=None, dk=None, dv=None, stream=None):
    """Gradients of attn_fwd_blocksparse_dropout's output (same mask, causal
    flag, p_drop, seed, offset).  Returns (dq, dk, dv)."""
    return _bwd_blocksparse("attn_bwd_blocksparse_dropout", q, k, v, o, do, lse, block_mask, scale, causal,
                            dq, dk, dv, stream, (p_drop, seed, offset))


def attn_fwd_fp8(q, k, v, descale_q, descale_k, descale_v, scale=None, causal=False, o=None, lse=None,
                 stream=None):
    """Forward with e4m3 inputs (torch.float8_e4m3fn or uint8 views) and
    per-tensor descale factors.  Returns (o bf16, lse fp32)."""
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    B, H, N, d = (int(x) for x in q.shape)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(name, t, q)
        if t.element_size() != 1:
            raise TypeError("%s must hold one-byte e4m3 values" % name)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q.device) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check("o", o, None, torch.bfloat16)
    _check("lse", lse, None, torch.float32)
    with _on_device(q):
        rc = lib().attn_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), float(descale_q), float(descale_k),
                                float(descale_v), o.data_ptr(), lse.data_ptr(), B, H, N, d, float(scale),
                                int(bool(causal)), _stream_handle(stream))
    if rc:
        raise AttnError("attn_fwd_fp8", rc)
    return o, lse


class _Attention(torch.autograd.Function):
    """Differentiable exact attention: forward through attn_fwd (or its
    dropout / block-mask variants), backward through the matching attn_bwd*
    from the saved O and LSE (P is recomputed, never stored)."""

    @staticmethod
    def forward(ctx, q, k, v, scale, causal, p_drop, seed, offset, block_mask):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        if block_mask is not None and p_drop > 0.0:
            o, lse = attn_fwd_blocksparse_dropout(q, k, v, block_mask, p_drop, seed, offset, scale=scale,
                                                  causal=causal)
        elif block_mask is not None:
            o, lse = attn_fwd_blocksparse(q, k, v, block_mask, scale=scale, causal=causal)
        elif p_drop > 0.0:
            o, lse = attn_fwd_dropout(q, k, v, p_drop, seed, offset, scale=scale, causal=causal)
        else:
            o, lse = attn_fwd(q, k, v, scale=scale, causal=causal)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.args = (scale, causal, p_drop, seed, offset, block_mask)
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        scale, causal, p_drop, seed, offset, block_mask = ctx.args
        do = do.contiguous()
        if block_mask is not None and p_drop > 0.0:
            dq, dk, dv = attn_bwd_blocksparse_dropout(q, k, v, o, do, lse, block_mask, p_drop, seed, offset,
                                                      scale=scale, causal=causal)
        elif block_mask is not None:
            dq, dk, dv = attn_bwd_blocksparse(q, k, v, o, do, lse, block_mask, scale=scale, causal=causal)
        elif p_drop > 0.0:
            dq, dk, dv = attn_bwd_dropout(q, k, v, o, do, lse, p_drop, seed, offset, scale=scale, causal=causal)
        else:
            dq, dk, dv = attn_bwd(q, k, v, o, do, lse, scale=scale, causal=causal)
        return dq, dk, dv, None, None, None, None, None, None


def attention(q, k, v, scale=None, causal=False, dropout_p=0.0, seed=0, offset=0, block_mask=None):
    """O = softmax(scale q k^T [+ causal mask]) v as a differentiable op on
    [B, H, N, d] CUDA tensors (bf16 or fp16).  Gradients flow to q, k and v
    through the recomputation backward.  With dropout_p > 0 the keep
    decisions come from (seed, offset); use a new offset per step.  With a
    block_mask (uint8 [H or 1, ceil(N/128), ceil(N/128)] on the device) only
    the enabled 128 x 128 tiles are computed, as in attn_fwd_blocksparse."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    return _Attention.apply(q, k, v, float(scale), bool(causal), float(dropout_p), int(seed), int(offset),
                            block_mask)


def sync_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the sticky device status."""
    return lib().attn_sync_status(_stream_handle(stream))

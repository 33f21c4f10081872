"""attn_bwd_noalloc: the backward for callers that must not allocate device
memory during the call (an allocator that must not be re-entered, a frozen
memory budget, a host that only hands over the tensors).  It is checked
through the C ABI against attn_bwd on the same inputs, on two calls in a row
with different problems (so a call cannot lean on scratch contents an earlier
call left behind); at the largest problem its fixed scratch array holds and
the smallest one it does not (the size rule of attn.h); and for the property
that defines it: the device's default memory pool, which the stream-ordered
allocator of attn_bwd draws from, sees no allocation during the call.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test."""
import ctypes
import math

import pytest
import torch

from io_aware_exact_12_gb300.synth import AttnShape, make_inputs

pytestmark = pytest.mark.gpu

TOL_GRAD = 2e-2  # the relative Frobenius tolerance the other gradient tests use
SCRATCH_BYTES = (32 << 20) + (512 << 10)  # the array's size, attn.h


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from io_aware_exact_12_gb300 import build as b
    b.build()
    import io_aware_exact_12_gb300 as pkg
    lib = pkg.lib()
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, F, I, P]
    lib.attn_bwd_noalloc.restype = I
    return lib


def _scratch_bytes(B, H, N, d):
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    return up(4 * B * H * N * d) + 2 * up(4 * B * H * ((N + 127) // 128) * 128)


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm().clamp_min(1e-30))


def _run(L, shape, seed, causal):
    import io_aware_exact_12_gb300 as pkg
    x = make_inputs(shape, "bf16", seed=seed, device="cuda")
    scale = 1.0 / math.sqrt(shape.d)
    o, lse = pkg.attn_fwd(x["q"], x["k"], x["v"], scale=scale, causal=causal)
    ref = pkg.attn_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, scale=scale, causal=causal)
    out = [torch.empty_like(x["q"]) for _ in range(3)]
    stream = torch.cuda.current_stream().cuda_stream
    rc = L.attn_bwd_noalloc(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(), o.data_ptr(),
                            x["do"].data_ptr(), lse.data_ptr(), out[0].data_ptr(), out[1].data_ptr(),
                            out[2].data_ptr(), shape.B, shape.H, shape.N, shape.d, scale, int(causal), stream)
    assert rc == 0, pkg.status_string(rc)
    assert pkg.sync_status() == 0
    for name, got, want in zip(("dq", "dk", "dv"), out, ref):
        assert torch.isfinite(got.float()).all(), name
        e = _rel(got, want)
        assert e <= TOL_GRAD, "%s: relative Frobenius difference %g" % (name, e)


def test_noalloc_matches_attn_bwd_on_two_calls_in_a_row(L):
    first = AttnShape(2, 4, 1000, 128)   # ragged N, head dim 128, causal
    second = AttnShape(1, 6, 700, 64)    # a different shape and mask on the same scratch
    assert _scratch_bytes(first.B, first.H, first.N, first.d) <= SCRATCH_BYTES
    _run(L, first, seed=31, causal=True)
    _run(L, second, seed=32, causal=False)


def test_noalloc_at_the_largest_problem_that_fits(L):
    largest = AttnShape(1, 8, 8192, 128)
    assert _scratch_bytes(largest.B, largest.H, largest.N, largest.d) == SCRATCH_BYTES  # fills the array exactly
    _run(L, largest, seed=33, causal=False)


@pytest.mark.parametrize("B,H,N,d", [(1, 8, 8193, 128),   # one row more than the largest that fits
                                     (1, 16, 8192, 128)])  # about twice the array
def test_noalloc_rejects_problems_beyond_its_scratch(L, B, H, N, d):
    assert _scratch_bytes(B, H, N, d) > SCRATCH_BYTES
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    span = 64 << 20  # far enough apart that no two of these (at most 33.6 MB) ranges overlap
    ptrs = [t.data_ptr() + span * i for i in range(5)]  # validated only, never dereferenced
    outs = [t.data_ptr() + span * (5 + i) for i in range(3)]
    lse_p = t.data_ptr() + span * 9
    rc = L.attn_bwd_noalloc(*ptrs, lse_p, *outs, B, H, N, d, 0.088, 1,
                            torch.cuda.current_stream().cuda_stream)
    assert rc == 2  # ATTN_ERR_UNSUPPORTED, nothing enqueued
    torch.cuda.synchronize()


def _cudart():
    """The CUDA runtime library the process has loaded (the one libattn.so uses)."""
    with open("/proc/self/maps") as f:
        for line in f:
            path = line.split()[-1]
            if "libcudart.so" in path:
                return ctypes.CDLL(path)
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            pass
    pytest.skip("CUDA runtime library not found")


USED_MEM_HIGH = 8  # cudaMemPoolAttrUsedMemHigh


def test_noalloc_allocates_nothing(L):
    """The stream-ordered allocator (cudaMallocAsync) serves from the device's
    default memory pool; its used-memory high-water mark, reset to zero, stays
    at zero across attn_bwd_noalloc and rises across attn_bwd (the positive
    control, which takes its scratch from that pool)."""
    import io_aware_exact_12_gb300 as pkg
    rt = _cudart()
    pool = ctypes.c_void_p()
    assert rt.cudaDeviceGetDefaultMemPool(ctypes.byref(pool), torch.cuda.current_device()) == 0

    def reset_high():
        assert rt.cudaMemPoolSetAttribute(pool, USED_MEM_HIGH, ctypes.byref(ctypes.c_uint64(0))) == 0

    def high():
        v = ctypes.c_uint64(0)
        assert rt.cudaMemPoolGetAttribute(pool, USED_MEM_HIGH, ctypes.byref(v)) == 0
        return v.value

    shape = AttnShape(1, 4, 1024, 64)
    x = make_inputs(shape, "bf16", seed=34, device="cuda")
    scale = 1.0 / math.sqrt(shape.d)
    o, lse = pkg.attn_fwd(x["q"], x["k"], x["v"], scale=scale, causal=True)
    out = [torch.empty_like(x["q"]) for _ in range(3)]
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    reset_high()
    rc = L.attn_bwd_noalloc(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(), o.data_ptr(),
                            x["do"].data_ptr(), lse.data_ptr(), out[0].data_ptr(), out[1].data_ptr(),
                            out[2].data_ptr(), shape.B, shape.H, shape.N, shape.d, scale, 1, stream)
    assert rc == 0
    assert pkg.sync_status() == 0
    assert high() == 0, "attn_bwd_noalloc drew %d bytes from the memory pool" % high()
    ref = pkg.attn_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, scale=scale, causal=True)
    torch.cuda.synchronize()
    assert high() > 0  # attn_bwd's scratch came from the same pool
    for name, got, want in zip(("dq", "dk", "dv"), out, ref):
        assert _rel(got, want) <= TOL_GRAD, name

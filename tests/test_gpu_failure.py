"""Device-side failure path: a bounded wait on a barrier that nothing arrives
on gives up, reports ATTN_ERR_TIMEOUT through the sticky status, clears, and
leaves the context usable (a normal forward still runs and matches the
oracle).  No GPU is made to fault, trap or hang."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_12_gb300.synth import AttnShape, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from io_aware_exact_12_gb300 import build as b
    b.build()
    import io_aware_exact_12_gb300 as p
    L = p.lib()
    L.attn_debug_wait_timeout.argtypes = [ctypes.c_int, ctypes.c_void_p]
    L.attn_debug_wait_timeout.restype = ctypes.c_int
    return p


def test_bounded_wait_reports_timeout_and_context_survives(pkg):
    L = pkg.lib()
    stream = torch.cuda.current_stream().cuda_stream
    assert pkg.sync_status() == 0
    assert L.attn_debug_wait_timeout(0, stream) == 1          # invalid limit, nothing enqueued
    assert L.attn_debug_wait_timeout(20000, stream) == 0      # 20 ms limit
    assert pkg.sync_status() == 4                              # ATTN_ERR_TIMEOUT
    assert pkg.sync_status() == 0                              # cleared
    x = make_inputs(AttnShape(1, 2, 300, 64), "bf16", seed=3)
    o, lse = pkg.attn_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), scale=0.125, causal=True)
    assert pkg.sync_status() == 0
    oo, lo = oracle.forward(x["q"].double().numpy(), x["k"].double().numpy(), x["v"].double().numpy(),
                            0.125, True)
    assert np.abs(lse.double().cpu().numpy() - lo).max() <= 1e-3
    assert np.abs(o.double().cpu().numpy() - oo).max() <= 2e-2

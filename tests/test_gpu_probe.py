"""The exponential-unit probe behind the C ABI (attn_probe_ex2): every thread's
8 recurrences x <- 2^x - 1.5 converge to the fixed point x = -1 (2^-1 - 1.5 =
-1, slope 0.35 < 1 there), so each output is -8 up to ex2.approx's error, and
every launched thread wrote its slot."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from io_aware_exact_12_gb300 import build as b
    b.build()
    yield


@pytest.mark.parametrize("blocks,iters", [(1, 1), (3, 64), (152 * 8, 256)])
def test_probe_writes_every_thread_and_converges(blocks, iters):
    import io_aware_exact_12_gb300 as attn
    sink = torch.full((blocks * attn.EX2_PROBE_THREADS + 5,), float("nan"), device="cuda")
    n = attn.probe_ex2(sink, blocks, iters)
    torch.cuda.synchronize()
    assert attn.sync_status() == 0
    assert n == blocks * 256 * iters * 8
    out = sink[: blocks * 256]
    assert torch.isfinite(out).all()
    assert torch.isnan(sink[blocks * 256:]).all()  # nothing written past the launched threads
    if iters >= 64:
        assert (out + 8.0).abs().max().item() < 1e-3
    else:
        assert ((out > -8.7) & (out < -7.9)).all()


def test_probe_rejects_a_short_sink():
    import io_aware_exact_12_gb300 as attn
    with pytest.raises(ValueError):
        attn.probe_ex2(torch.empty(255, device="cuda"), 1, 1)

"""The differentiable wrapper gives exactly what the C entry points give:
O from attn_fwd and, through loss.backward(), the gradients of attn_bwd
(and of the dropout and block-mask pairs), bit for bit."""
import math

import pytest
import torch

from io_aware_exact_12_gb300.synth import AttnShape, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from io_aware_exact_12_gb300 import build as b
    b.build()
    import io_aware_exact_12_gb300 as p
    p.lib()
    return p


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("p_drop", [0.0, 0.2])
def test_autograd_matches_the_entry_points(pkg, causal, p_drop):
    x = make_inputs(AttnShape(2, 3, 300, 64), "bf16", seed=31)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    s = 1 / math.sqrt(64)
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = pkg.attention(qq, kk, vv, scale=s, causal=causal, dropout_p=p_drop, seed=7, offset=3)
    (o.float() * do.float()).sum().backward()
    if p_drop > 0:
        o_ref, lse = pkg.attn_fwd_dropout(q, k, v, p_drop, 7, 3, scale=s, causal=causal)
        g = pkg.attn_bwd_dropout(q, k, v, o_ref, do, lse, p_drop, 7, 3, scale=s, causal=causal)
    else:
        o_ref, lse = pkg.attn_fwd(q, k, v, scale=s, causal=causal)
        g = pkg.attn_bwd(q, k, v, o_ref, do, lse, scale=s, causal=causal)
    assert pkg.sync_status() == 0
    assert torch.equal(o.detach(), o_ref)
    # dK and dV bit for bit; dQ is reduced with atomics in any order
    assert torch.equal(kk.grad, g[1]) and torch.equal(vv.grad, g[2])
    assert (qq.grad.float() - g[0].float()).abs().max().item() <= 1e-2 * g[0].float().abs().max().item()


@pytest.mark.parametrize("p_drop", [0.0, 0.3])
def test_autograd_with_a_block_mask(pkg, p_drop):
    x = make_inputs(AttnShape(1, 2, 700, 128), "bf16", seed=33)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    g0 = torch.Generator().manual_seed(2)
    mask = (torch.rand((2, 6, 6), generator=g0) < 0.5).to(torch.uint8)
    mask[:, torch.arange(6), torch.arange(6)] = 1
    mask = mask.cuda()
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = pkg.attention(qq, kk, vv, scale=0.09, causal=True, dropout_p=p_drop, seed=11, offset=5, block_mask=mask)
    (o.float() * do.float()).sum().backward()
    if p_drop > 0:
        o_ref, lse = pkg.attn_fwd_blocksparse_dropout(q, k, v, mask, p_drop, 11, 5, scale=0.09, causal=True)
        g = pkg.attn_bwd_blocksparse_dropout(q, k, v, o_ref, do, lse, mask, p_drop, 11, 5, scale=0.09, causal=True)
    else:
        o_ref, lse = pkg.attn_fwd_blocksparse(q, k, v, mask, scale=0.09, causal=True)
        g = pkg.attn_bwd_blocksparse(q, k, v, o_ref, do, lse, mask, scale=0.09, causal=True)
    assert pkg.sync_status() == 0
    assert torch.equal(o.detach(), o_ref)
    assert torch.equal(kk.grad, g[1]) and torch.equal(vv.grad, g[2])
    assert (qq.grad.float() - g[0].float()).abs().max().item() <= 1e-2 * g[0].float().abs().max().item()

"""Decode (one query token per (batch, head) against a KV cache of L tokens)
against the float64 oracle.  The oracle's per-row entry point computes the
plain definition for the query placed at row L-1 of an L-row problem with no
mask, i.e. attention of that query over all L keys.  Tolerances are the
forward's: max |dO| <= 1e-2 beyond the output type's own rounding, max
|dLSE| <= 1e-3."""
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
    p.lib()
    return p


def _half_ulp_bf16(ref):
    e = np.floor(np.log2(np.maximum(np.abs(ref), 1e-30)))
    return np.exp2(e - 8)


def _oracle_decode(q, k, v, scale, heads):
    """q: [BH, d], k/v: [BH, L, d] float64 -> (o [n, d], lse [n]) for the listed heads."""
    L, d = k.shape[1], k.shape[2]
    os_, ls = [], []
    for h in heads:
        qf = np.zeros((1, 1, L, d))
        qf[0, 0, L - 1] = q[h]
        o, lse, _ = oracle.rows(qf, k[h][None, None], v[h][None, None], None, scale, False,
                                np.array([0]), np.array([L - 1]))
        os_.append(o[0])
        ls.append(lse[0])
    return np.array(os_), np.array(ls)


def _run(pkg, B, H, L, d, scale, seed, heads=None):
    kv = make_inputs(AttnShape(B, H, L, d), "bf16", seed=seed, with_grad=False)
    q = make_inputs(AttnShape(B, H, 1, d), "bf16", seed=seed + 1000, with_grad=False)["q"]
    o, lse = pkg.attn_decode(q.cuda(), kv["k"].cuda(), kv["v"].cuda(), scale=scale)
    assert pkg.sync_status() == 0
    assert pkg.last_launch_count() == 2
    BH = B * H
    heads = list(range(BH)) if heads is None else heads
    qd = q.double().numpy().reshape(BH, d)
    kd = kv["k"].double().numpy().reshape(BH, L, d)
    vd = kv["v"].double().numpy().reshape(BH, L, d)
    ro, rl = _oracle_decode(qd, kd, vd, scale, heads)
    go = o.double().cpu().numpy().reshape(BH, d)[heads]
    gl = lse.double().cpu().numpy().reshape(BH)[heads]
    err = np.abs(go - ro)
    assert (err - _half_ulp_bf16(ro)).max() <= 1e-2, "max|dO| %g" % err.max()
    assert np.abs(gl - rl).max() <= 1e-3, "max|dLSE| %g" % np.abs(gl - rl).max()
    return o, lse, q, kv


@pytest.mark.parametrize("L", [1, 2, 7, 255, 1000, 4097])
@pytest.mark.parametrize("d", [32, 64, 128])
def test_decode_matches_oracle(pkg, L, d):
    _run(pkg, 2, 3, L, d, 1.0 / math.sqrt(d), seed=L * 3 + d)


def test_decode_single_key_closed_form(pkg):
    """L = 1: O = v_0 exactly and LSE = scale q.k_0."""
    o, lse, q, kv = _run(pkg, 2, 4, 1, 128, 0.09, seed=5)
    assert torch.equal(o.cpu(), kv["v"][:, :, 0])
    ref = 0.09 * (q[:, :, 0].double() * kv["k"][:, :, 0].double()).sum(-1)
    assert (lse.double().cpu() - ref).abs().max().item() <= 1e-4


@pytest.mark.parametrize("scale", [0.0, -0.3, 0.5])
def test_decode_scales(pkg, scale):
    _run(pkg, 1, 4, 3000, 128, scale, seed=9)


def test_decode_long_cache_sampled_heads(pkg):
    """A 32768-token cache over 64 heads (many splits per head), 6 heads checked."""
    _run(pkg, 4, 16, 32768, 128, 1.0 / math.sqrt(128), seed=11, heads=[0, 1, 17, 33, 62, 63])


def test_decode_equals_last_row_of_causal_forward(pkg):
    """Decoding the last token equals the last row of the causal forward."""
    B, H, L, d = 1, 4, 777, 64
    x = make_inputs(AttnShape(B, H, L, d), "bf16", seed=21, with_grad=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o_f, l_f = pkg.attn_fwd(q, k, v, scale=0.125, causal=True)
    o_d, l_d = pkg.attn_decode(q[:, :, L - 1].contiguous(), k, v, scale=0.125)
    assert pkg.sync_status() == 0
    assert (o_f[:, :, L - 1].float() - o_d.float()).abs().max().item() <= 2e-2
    assert (l_f[:, :, L - 1] - l_d).abs().max().item() <= 1e-3

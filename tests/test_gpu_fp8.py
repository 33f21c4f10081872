"""FP8 (e4m3) forward against the float64 oracle evaluated on the exact real
inputs descale * e4m3.

Tolerance, derived from the arithmetic: the kernel rounds each weight P_ij
to e4m3 (relative error <= 2^-4 in the normal range) and normalises O by the
sum of the rounded weights, so O_gpu - O = sum_j (w~_j - w_j)(v_j - O) with
|w~_j - w_j| <= w_j * 2 * 2^-4 / (1 - 2^-4); hence
    |dO_ic| <= 0.134 * sum_j P_ij |V_jc - O_ic|  + 1/2 ulp of the bf16 output + 2e-3
(the last term covers fp32 accumulation, exp2 and weights rounded in e4m3's
subnormal range).  LSE uses the exact fp32 sum: |dLSE| <= 1e-3."""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_12_gb300.synth import AttnShape, dequantize_e4m3, make_inputs_fp8

pytestmark = pytest.mark.gpu

REL_W = 2 * 2.0 ** -4 / (1 - 2.0 ** -4) + 1e-3


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


def _gpu(pkg, x, scale, causal):
    q8, k8, v8 = (x[n][0].cuda() for n in ("q", "k", "v"))
    o, lse = pkg.attn_fwd_fp8(q8, k8, v8, x["q"][1], x["k"][1], x["v"][1], scale=scale, causal=causal)
    assert pkg.sync_status() == 0
    return o, lse


def _bound(P, V, O):
    """0.134 * sum_j P_ij |V_jc - O_ic| for one head, in row chunks."""
    out = np.empty_like(O)
    for r0 in range(0, O.shape[0], 64):
        r1 = min(r0 + 64, O.shape[0])
        out[r0:r1] = REL_W * np.einsum("ij,ijc->ic", P[r0:r1], np.abs(V[None, :, :] - O[r0:r1, None, :]))
    return out


def _check_full(pkg, shape, seed, causal, qk_std=1.0, scale=None):
    x = make_inputs_fp8(shape, seed=seed, qk_std=qk_std)
    scale = 1.0 / math.sqrt(shape.d) if scale is None else scale
    o, lse = _gpu(pkg, x, scale, causal)
    q, k, v = (dequantize_e4m3(*x[n]).numpy() for n in ("q", "k", "v"))
    oo, lo, P = oracle.forward(q, k, v, scale, causal, want_p=True)
    go = o.double().cpu().numpy()
    err = np.abs(go - oo)
    for b in range(shape.B):
        for h in range(shape.H):
            allow = _bound(P[b, h], v[b, h], oo[b, h]) + _half_ulp_bf16(oo[b, h]) + 2e-3
            worst = (err[b, h] - allow).max()
            assert worst <= 0, "head (%d,%d): |dO| exceeds the derived bound by %g" % (b, h, worst)
    assert np.abs(lse.double().cpu().numpy() - lo).max() <= 1e-3
    rel = np.linalg.norm(go - oo) / np.linalg.norm(oo)
    return rel


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 77, 300, 1024])
def test_fp8_forward_matches_oracle(pkg, N, causal):
    _check_full(pkg, AttnShape(1, 2, N, 128), seed=N + 3, causal=causal)


def test_fp8_forward_logit_stress(pkg):
    _check_full(pkg, AttnShape(1, 2, 512, 128), seed=17, causal=True, qk_std=4.0, scale=0.125)


def test_fp8_forward_scale_zero(pkg):
    _check_full(pkg, AttnShape(1, 1, 200, 128), seed=19, causal=False, scale=0.0)


def test_fp8_causal_mask_bit_exact(pkg):
    shape = AttnShape(1, 2, 600, 128)
    x = make_inputs_fp8(shape, seed=23)
    o1, l1 = _gpu(pkg, x, 0.088, True)
    t = 333
    y = dict(x)
    for n in ("k", "v"):
        b = x[n][0].clone()
        b[:, :, t:] = 0x38  # e4m3 1.0
        y[n] = (b, x[n][1])
    o2, l2 = _gpu(pkg, y, 0.088, True)
    assert torch.equal(o1[:, :, :t], o2[:, :, :t]) and torch.equal(l1[:, :, :t], l2[:, :, :t])


def test_fp8_long_sequence_sampled(pkg):
    """B=2 H=16 N=8192 d=128 (the bench shape): LSE on sampled rows within 1e-3,
    O within the derived bound using the oracle's own probabilities."""
    shape = AttnShape(2, 16, 8192, 128)
    x = make_inputs_fp8(shape, seed=29)
    scale = 1.0 / math.sqrt(128)
    o, lse = _gpu(pkg, x, scale, False)
    q, k, v = (dequantize_e4m3(*x[n]).numpy() for n in ("q", "k", "v"))
    rng = np.random.default_rng(5)
    bh = rng.integers(0, 32, 64)
    ri = rng.integers(0, 8192, 64)
    ro, rl, _ = oracle.rows(q, k, v, None, scale, False, bh, ri)
    gl = lse.double().cpu().numpy().reshape(32, 8192)[bh, ri]
    assert np.abs(gl - rl).max() <= 1e-3
    go = o.double().cpu().numpy().reshape(32, 8192, 128)[bh, ri]
    qf, kf, vf = q.reshape(32, 8192, 128), k.reshape(32, 8192, 128), v.reshape(32, 8192, 128)
    for n in range(len(bh)):
        p = np.exp(scale * kf[bh[n]] @ qf[bh[n], ri[n]] - rl[n])  # the oracle's probabilities of this row
        allow = REL_W * (p[:, None] * np.abs(vf[bh[n]] - ro[n][None, :])).sum(0) + _half_ulp_bf16(ro[n]) + 2e-3
        assert (np.abs(go[n] - ro[n]) - allow).max() <= 0

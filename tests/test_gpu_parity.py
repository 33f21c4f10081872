"""GPU parity: the CUDA path (through the C ABI) against the float64 CPU
oracle on the same seeded inputs.

Tolerances (bf16/fp16 inputs, fp32 accumulation): max |dO| <= 1e-2 beyond
the rounding of the result to the output type itself (half an ulp of bf16 at
|O| in [4, 8) is 0.0156, so no bf16 output can meet a bare 1e-2 there),
max |dLSE| <= 1e-3, relative Frobenius error of dQ, dK, dV <= 2e-2; the
causal mask must hold bit-exactly (nothing behind the diagonal may change an
output).  Small configurations are compared in full; at N = 8192 and 32768
sampled rows (O, LSE, dQ) and sampled key columns (dK, dV) are compared, plus
properties that hold at any size.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_12_gb300.synth import AttnShape, make_inputs, sample_rows

pytestmark = pytest.mark.gpu

TOL_O = 1e-2
TOL_LSE = 1e-3
TOL_GRAD = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from io_aware_exact_12_gb300 import build as b
    b.build()
    import io_aware_exact_12_gb300 as pkg
    pkg.lib()
    yield


def _pkg():
    import io_aware_exact_12_gb300 as pkg
    return pkg


def gpu_fwd(x, scale, causal):
    pkg = _pkg()
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = pkg.attn_fwd(q, k, v, scale=scale, causal=causal)
    assert pkg.sync_status() == 0
    return o, lse


def gpu_bwd(x, o, lse, scale, causal):
    pkg = _pkg()
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    dq, dk, dv = pkg.attn_bwd(q, k, v, o, do, lse, scale=scale, causal=causal)
    assert pkg.sync_status() == 0
    return dq, dk, dv


def f64(t):
    return t.detach().double().cpu().numpy()


def rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def half_ulp(ref, dtype):
    """Half a unit in the last place of the output format at the exact value:
    the closest any bf16/fp16 output can be to the float64 answer."""
    e = np.floor(np.log2(np.maximum(np.abs(ref), 1e-30)))
    if dtype == torch.bfloat16:
        return np.exp2(e - 8)
    return np.exp2(np.maximum(e, -14) - 11)


def check_o(o, ref):
    """max |dO| <= 1e-2 on top of the unavoidable rounding of the result to
    the output type (half an ulp at the exact value)."""
    err = np.abs(f64(o) - ref)
    excess = (err - half_ulp(ref, o.dtype)).max()
    assert excess <= TOL_O, "max|dO| beyond output rounding = %g (raw max %g)" % (excess, err.max())
    return err.max()


def check_fwd_full(x, scale, causal, o, lse):
    oo, lo = oracle.forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale, causal)
    check_o(o, oo)
    el = np.abs(f64(lse) - lo).max()
    assert el <= TOL_LSE, "max|dLSE| = %g" % el
    return oo, lo


def check_bwd_full(x, scale, causal, oo, grads):
    dq, dk, dv = oracle.backward(f64(x["q"]), f64(x["k"]), f64(x["v"]), oo, f64(x["do"]), scale, causal)
    # Where an exact gradient vanishes identically (N = 1: dQ = dK = 0) a relative
    # error is undefined; the denominator is then floored at 1e-3 |dO|.
    floor = 1e-3 * float(np.linalg.norm(f64(x["do"])))
    for name, g, ref in (("dq", grads[0], dq), ("dk", grads[1], dk), ("dv", grads[2], dv)):
        e = float(np.linalg.norm(f64(g) - ref) / max(np.linalg.norm(ref), floor))
        assert e <= TOL_GRAD, "%s rel Frobenius error %g" % (name, e)


# ------------------------------------------------------------------ configs
# 1: causal fwd+bwd, B=2 H=4 N=64 d=32 bf16, scale 1/sqrt(32)
@pytest.mark.parametrize("causal", [True, False])
def test_c1_small_fwd_bwd(causal):
    x = make_inputs(AttnShape(2, 4, 64, 32), "bf16", seed=1)
    s = 1.0 / math.sqrt(32)
    o, lse = gpu_fwd(x, s, causal)
    oo, _ = check_fwd_full(x, s, causal, o, lse)
    check_bwd_full(x, s, causal, oo, gpu_bwd(x, o, lse, s, causal))


# 2: fp16 fwd, B=2 H=8 N=512 d=64, scale 1/8, causal and not; N=500 exercises a ragged tile
@pytest.mark.parametrize("N", [512, 500])
@pytest.mark.parametrize("causal", [True, False])
def test_c2_fp16_fwd(N, causal):
    x = make_inputs(AttnShape(2, 8, N, 64), "f16", seed=2)
    o, lse = gpu_fwd(x, 0.125, causal)
    check_fwd_full(x, 0.125, causal, o, lse)


@pytest.mark.parametrize("N", [512, 500])
def test_c2_fp16_bwd(N):
    x = make_inputs(AttnShape(2, 8, N, 64), "f16", seed=2)
    o, lse = gpu_fwd(x, 0.125, True)
    oo, _ = check_fwd_full(x, 0.125, True, o, lse)
    check_bwd_full(x, 0.125, True, oo, gpu_bwd(x, o, lse, 0.125, True))


# 3: GPT-2-small shape, B=8 H=12 N=1024 d=64 bf16 causal, plus logits spanning +-100
@pytest.mark.parametrize("qk_std", [1.0, 4.0])
def test_c3_gpt2_shape(qk_std):
    x = make_inputs(AttnShape(8, 12, 1024, 64), "bf16", seed=3, qk_std=qk_std)
    o, lse = gpu_fwd(x, 0.125, True)
    oo, _ = check_fwd_full(x, 0.125, True, o, lse)
    check_bwd_full(x, 0.125, True, oo, gpu_bwd(x, o, lse, 0.125, True))


def _check_sampled(x, scale, causal, o, lse, grads, nrows, heads_for_cols, ncols):
    shape = AttnShape(*x["q"].shape)
    q, k, v, do = (f64(x[n]) for n in ("q", "k", "v", "do"))
    bh, ri = sample_rows(shape, nrows, seed=11)
    ro, rl, rdq = oracle.rows(q, k, v, do, scale, causal, bh, ri)
    N, d = shape.N, shape.d
    go = f64(o).reshape(-1, N, d)[bh, ri]
    gl = f64(lse).reshape(-1, N)[bh, ri]
    gdq = f64(grads[0]).reshape(-1, N, d)[bh, ri]
    err = np.abs(go - ro)
    assert (err - half_ulp(ro, o.dtype)).max() <= TOL_O, "sampled max|dO| %g" % err.max()
    assert np.abs(gl - rl).max() <= TOL_LSE
    assert rel_fro(gdq, rdq) <= TOL_GRAD
    # sampled key columns: every row's LSE and D of the chosen heads from the oracle itself
    for h in heads_for_cols:
        all_rows = np.arange(N)
        fo, fl, _ = oracle.rows(q, k, v, None, scale, causal, np.full(N, h), all_rows)
        lse_all = np.zeros((shape.B * shape.H, N))
        D_all = np.zeros((shape.B * shape.H, N))
        lse_all[h] = fl
        D_all[h] = (do.reshape(-1, N, d)[h] * fo).sum(-1)
        cols = np.random.default_rng(h).choice(N, size=ncols, replace=False)
        cols[:2] = [0, N - 1]
        dk_ref, dv_ref = oracle.cols(q, k, v, do, lse_all.reshape(shape.B, shape.H, N),
                                     D_all.reshape(shape.B, shape.H, N), scale, causal,
                                     np.full(ncols, h), cols)
        gdk = f64(grads[1]).reshape(-1, N, d)[h, cols]
        gdv = f64(grads[2]).reshape(-1, N, d)[h, cols]
        assert rel_fro(gdk, dk_ref) <= TOL_GRAD, "dk head %d" % h
        assert rel_fro(gdv, dv_ref) <= TOL_GRAD, "dv head %d" % h


def _check_identities(x, grads):
    """sum_j dV_j = sum_i dO_i and sum_j dK_j = 0, per head (exact in exact arithmetic)."""
    dk = grads[1].float().sum(2)
    dv = grads[2].float().sum(2)
    dos = x["do"].cuda().float().sum(2)
    scale_v = grads[2].float().abs().sum(2).max().item()
    scale_k = grads[1].float().abs().sum(2).max().item()
    assert (dv - dos).abs().max().item() <= 1e-2 * max(scale_v, 1.0)
    assert dk.abs().max().item() <= 1e-2 * max(scale_k, 1.0)


# 4: long sequence, B=2 H=16 N=8192 d=128 bf16, causal and not
@pytest.mark.parametrize("causal", [True, False])
def test_c4_long_sequence(causal):
    x = make_inputs(AttnShape(2, 16, 8192, 128), "bf16", seed=4)
    s = 1.0 / math.sqrt(128)
    o, lse = gpu_fwd(x, s, causal)
    grads = gpu_bwd(x, o, lse, s, causal)
    _check_sampled(x, s, causal, o, lse, grads, nrows=512, heads_for_cols=[0, 11, 20, 31], ncols=64)
    _check_identities(x, grads)


# 5: very long single sequence, B=1 H=8 N=32768 d=128 bf16 causal; 512 sampled
# query rows (O, LSE, dQ) and 512 sampled key columns, 64 in each of the 8
# heads (dK, dV; the oracle streams every row's LSE and D of each head)
def test_c5_very_long_sequence():
    x = make_inputs(AttnShape(1, 8, 32768, 128), "bf16", seed=5)
    s = 1.0 / math.sqrt(128)
    o, lse = gpu_fwd(x, s, True)
    grads = gpu_bwd(x, o, lse, s, True)
    _check_sampled(x, s, True, o, lse, grads, nrows=512, heads_for_cols=list(range(8)), ncols=64)
    _check_identities(x, grads)


# The other compiled variants (fp16; d = 64 and 32) at a multi-wave size:
# N = 4096 (32 key tiles), 16 heads, sampled rows and key columns.
@pytest.mark.parametrize("dtype,d,causal", [("f16", 128, False), ("f16", 128, True), ("bf16", 64, False),
                                            ("bf16", 64, True), ("bf16", 32, True), ("f16", 32, False)])
def test_long_sequence_other_variants(dtype, d, causal):
    x = make_inputs(AttnShape(2, 8, 4096, d), dtype, seed=12)
    s = 1.0 / math.sqrt(d)
    o, lse = gpu_fwd(x, s, causal)
    grads = gpu_bwd(x, o, lse, s, causal)
    _check_sampled(x, s, causal, o, lse, grads, nrows=256, heads_for_cols=[0, 15], ncols=32)
    _check_identities(x, grads)


# The causal kernels visit blocks heaviest first within groups of heads.  The
# backward groups 32 MB / (8 N d bytes) heads: 4 at N = 8192, d = 128, so 10
# heads make groups of 4, 4 and 2; the forward groups 128 MB / (4 N d bytes):
# 8 at N = 32768, so 10 heads make 8 and 2.  Outputs are preset to NaN, so a
# block the order skipped would show; every row and key column is covered by
# the LSE finiteness and the per-head identities, sampled ones by the oracle.
@pytest.mark.parametrize("N", [8192, 32768])
def test_causal_order_short_last_head_group(N):
    pkg = _pkg()
    x = make_inputs(AttnShape(1, 10, N, 128), "bf16", seed=6)
    s = 1.0 / math.sqrt(128)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device="cuda")
    pkg.attn_fwd(q, k, v, scale=s, causal=True, o=o, lse=lse)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    pkg.attn_bwd(q, k, v, o, do, lse, scale=s, causal=True, dq=dq, dk=dk, dv=dv)
    assert pkg.sync_status() == 0
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t).all()
    grads = (dq, dk, dv)
    _check_sampled(x, s, True, o, lse, grads, nrows=256, heads_for_cols=[9], ncols=32)
    _check_identities(x, grads)


# The same with one-tile CTAs (d = 64): the forward groups 128 MB / (4 N d
# bytes) = 16 heads at N = 32768, so 20 heads make 16 and 4; the backward 2
# heads a group.
def test_causal_order_one_tile_ctas():
    pkg = _pkg()
    x = make_inputs(AttnShape(1, 20, 32768, 64), "bf16", seed=16)
    s = 1.0 / math.sqrt(64)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device="cuda")
    pkg.attn_fwd(q, k, v, scale=s, causal=True, o=o, lse=lse)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    pkg.attn_bwd(q, k, v, o, do, lse, scale=s, causal=True, dq=dq, dk=dk, dv=dv)
    assert pkg.sync_status() == 0
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t).all()
    grads = (dq, dk, dv)
    _check_sampled(x, s, True, o, lse, grads, nrows=256, heads_for_cols=[19], ncols=32)
    _check_identities(x, grads)


# ------------------------------------------------------------- edge cases
@pytest.mark.parametrize("N", [1, 2, 63, 127, 129, 255, 257, 383])
@pytest.mark.parametrize("d", [32, 64, 128])
def test_ragged_and_tiny(N, d):
    x = make_inputs(AttnShape(1, 3, N, d), "bf16", seed=N * 7 + d)
    s = 1.0 / math.sqrt(d)
    for causal in (False, True):
        o, lse = gpu_fwd(x, s, causal)
        oo, _ = check_fwd_full(x, s, causal, o, lse)
        check_bwd_full(x, s, causal, oo, gpu_bwd(x, o, lse, s, causal))


@pytest.mark.parametrize("scale", [0.0, -0.2, 1.7])
def test_unusual_scales(scale):
    x = make_inputs(AttnShape(1, 2, 200, 64), "bf16", seed=21)
    for causal in (False, True):
        o, lse = gpu_fwd(x, scale, causal)
        oo, _ = check_fwd_full(x, scale, causal, o, lse)
        check_bwd_full(x, scale, causal, oo, gpu_bwd(x, o, lse, scale, causal))


@pytest.mark.parametrize("scale", [1.0, 2.0])
def test_worked_example_on_gpu(scale):
    """Scores [90, 80, 70] in the first key tile and 95 at key 128 (second tile):
    the later, larger score forces the correction the pages describe (at
    scale 2 the max grows by 10, past the kernel's lazy-rescale threshold)."""
    N, d = 256, 32
    q = torch.zeros(1, 1, N, d)
    q[..., 0] = 1.0
    k = torch.zeros(1, 1, N, d)
    k[..., 0] = -9984.0  # exact in bf16; exp of it is 0
    for j, sc in ((0, 90.0), (1, 80.0), (2, 70.0), (128, 95.0)):
        k[0, 0, j, 0] = sc
    v = torch.randn(1, 1, N, d, generator=torch.Generator().manual_seed(0))
    x = {"q": q.bfloat16(), "k": k.bfloat16(), "v": v.bfloat16()}
    o, lse = gpu_fwd(x, scale, False)
    check_fwd_full(x, scale, False, o, lse)
    ell = sum(math.exp(scale * (t - 95.0)) for t in (90.0, 80.0, 70.0, 95.0))
    assert abs(lse[0, 0, 0].item() - (scale * 95.0 + math.log(ell))) <= TOL_LSE


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_constant_v(d, causal):
    """Every row of V equal to one vector c (per head): the weights of a row sum
    to 1, so O_i = c exactly for every row; and dP_ij = dO_i . c = D_i for every
    key, so dS = 0 and dQ = dK = 0 exactly (only rounding remains), while
    dV = P^T dO is unchanged in form."""
    B, H, N = 2, 2, 300
    x = make_inputs(AttnShape(B, H, N, d), "bf16", seed=8 + d)
    c = torch.randn(B, H, 1, d, generator=torch.Generator().manual_seed(d)).bfloat16()
    s = 1.0 / math.sqrt(d)
    grads_random_v = gpu_bwd(x, *gpu_fwd(x, s, causal), s, causal)
    x["v"] = c.expand(B, H, N, d).contiguous()
    o, lse = gpu_fwd(x, s, causal)
    check_o(o, np.broadcast_to(f64(c), (B, H, N, d)))
    oo, _ = check_fwd_full(x, s, causal, o, lse)
    dq, dk, dv = gpu_bwd(x, o, lse, s, causal)
    for name, g, ref in (("dq", dq, grads_random_v[0]), ("dk", dk, grads_random_v[1])):
        ratio = float(g.float().norm() / ref.float().norm())
        assert ratio <= TOL_GRAD, "%s is %g of its size with a random V" % (name, ratio)
    _, _, dv_ref = oracle.backward(f64(x["q"]), f64(x["k"]), f64(x["v"]), oo, f64(x["do"]), s, causal)
    assert rel_fro(f64(dv), dv_ref) <= TOL_GRAD


# ----------------------------------------------------- causal bit-exactness
def test_causal_mask_is_bit_exact():
    N, t = 1000, 613
    x = make_inputs(AttnShape(1, 4, N, 64), "bf16", seed=9)
    o1, l1 = gpu_fwd(x, 0.125, True)
    y = dict(x)
    y["k"] = x["k"].clone()
    y["v"] = x["v"].clone()
    y["k"][:, :, t:] = 3.0
    y["v"][:, :, t:] = -7.0
    o2, l2 = gpu_fwd(y, 0.125, True)
    assert torch.equal(o1[:, :, :t], o2[:, :, :t])
    assert torch.equal(l1[:, :, :t], l2[:, :, :t])
    # gradients of keys/values at >= t do not depend on dO rows < t
    g1 = gpu_bwd(x, o1, l1, 0.125, True)
    z = dict(x)
    z["do"] = x["do"].clone()
    z["do"][:, :, :t] = 5.0
    g2 = gpu_bwd(z, o1, l1, 0.125, True)
    assert torch.equal(g1[1][:, :, t:], g2[1][:, :, t:])
    assert torch.equal(g1[2][:, :, t:], g2[2][:, :, t:])


def test_forward_is_deterministic():
    x = make_inputs(AttnShape(2, 4, 777, 128), "bf16", seed=10)
    o1, l1 = gpu_fwd(x, 0.09, True)
    o2, l2 = gpu_fwd(x, 0.09, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d,causal", [(128, False), (128, True), (64, False), (32, True)])
def test_repeated_runs_bit_identical(d, causal):
    """The next S is issued right behind the MMA that reads the TMEM columns it
    overwrites (P V in the forward at d = 128, dV in the backward), relying on
    the tensor pipe executing one thread's MMAs in issue order.  Were that
    order ever broken, P (or P^T) would be overwritten while being read, with a
    timing-dependent result: over a grid of several waves, repeated runs must
    agree bit for bit in O, LSE, dK and dV (dQ is reduced in arbitrary order),
    and the first run must match the oracle on sampled rows and columns."""
    x = make_inputs(AttnShape(2, 8, 2048, d), "bf16", seed=21 + d)
    s = 1.0 / math.sqrt(d)
    o0, l0 = gpu_fwd(x, s, causal)
    g0 = gpu_bwd(x, o0, l0, s, causal)
    for _ in range(6):
        o, l = gpu_fwd(x, s, causal)
        assert torch.equal(o, o0) and torch.equal(l, l0)
    for _ in range(3):
        g = gpu_bwd(x, o0, l0, s, causal)
        assert torch.equal(g[1], g0[1]) and torch.equal(g[2], g0[2])
    _check_sampled(x, s, causal, o0, l0, g0, nrows=64, heads_for_cols=[0, 15], ncols=16)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance_on_gpu(causal):
    """Adding one vector c to every key adds scale * q_i . c to every score of
    row i, which the softmax removes: O is unchanged and LSE_i moves by
    scale * q_i . c.  K is put on a grid of 1/16 in [-4, 4) so that K + 1/2 is
    exact in bf16 (at most 7 significant bits); both runs are compared with
    each other and with the oracle of the unshifted problem."""
    x = make_inputs(AttnShape(1, 2, 256, 64), "bf16", seed=12)
    x["k"] = ((x["k"].float() * 16).round().clamp(-64, 63) / 16).bfloat16()
    shifted = x["k"].float() + 0.5
    assert torch.equal(shifted.bfloat16().float(), shifted)  # the shift is exact
    y = dict(x)
    y["k"] = shifted.bfloat16()
    o1, l1 = gpu_fwd(x, 0.125, causal)
    o2, l2 = gpu_fwd(y, 0.125, causal)
    oo, lo = oracle.forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), 0.125, causal)
    check_o(o1, oo)
    check_o(o2, oo)  # the shifted problem has the same exact O
    assert (o1.float() - o2.float()).abs().max().item() <= 2 * TOL_O
    lse_shift = 0.125 * 0.5 * f64(x["q"]).sum(-1)
    assert np.abs(f64(l2) - f64(l1) - lse_shift).max() <= 2 * TOL_LSE
    assert np.abs(f64(l2) - (lo + lse_shift)).max() <= TOL_LSE


def test_launch_count_and_status():
    pkg = _pkg()
    x = make_inputs(AttnShape(1, 1, 128, 64), "bf16", seed=13)
    o, lse = gpu_fwd(x, 0.125, False)
    assert pkg.last_launch_count() == 1
    gpu_bwd(x, o, lse, 0.125, False)
    assert pkg.last_launch_count() == 3
    assert pkg.sync_status() == 0

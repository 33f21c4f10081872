"""Pins for the float64 CPU oracle (no GPU needed).

The oracle is checked against things other than itself: the worked example
printed on the pages, closed forms, invariants of softmax attention, central
finite differences of its own forward pass (which pin the analytic backward),
and an independently written blockwise online-softmax reference.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle.blockwise import attention_blockwise, attention_blockwise_bhnd
from io_aware_exact_12_gb300.synth import AttnShape, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_worked_example():
    vals = {}
    with open(os.path.join(GOLDEN, "worked_example.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rhs = (t.strip() for t in line.split("="))
            vals[key] = [float(x) for x in rhs.split()]
    return vals


def _np_inputs(B, H, N, d, dtype="bf16", seed=0, qk_std=1.0):
    t = make_inputs(AttnShape(B, H, N, d), dtype=dtype, seed=seed, qk_std=qk_std)
    return {k: v.double().numpy() for k, v in t.items()}


# ---------------------------------------------------------------- (b) worked example
def test_worked_example_closed_form():
    """Scores [90, 80, 70 | 95] realised with d = 1, q = 1, k_j = score_j, scale = 1."""
    ex = _load_worked_example()
    scores = ex["block1"] + ex["block2"]
    n = len(scores)
    q = np.ones((1, 1, n, 1))
    k = np.array(scores, dtype=np.float64).reshape(1, 1, n, 1)
    v = np.arange(1.0, n + 1.0).reshape(1, 1, n, 1)
    o, lse, p = oracle.forward(q, k, v, 1.0, False, want_p=True)
    m = ex["final_max"][0]
    # closed form: l = sum_j e^(x_j - 95) = 1 + e^-5 + e^-15 + e^-25
    ell = 1.0 + math.exp(-5.0) + math.exp(-15.0) + math.exp(-25.0)
    for i in range(n):
        for j, x in enumerate(scores):
            assert p[0, 0, i, j] == pytest.approx(math.exp(x - m) / ell, rel=1e-14, abs=1e-300)
        assert lse[0, 0, i] == pytest.approx(m + math.log(ell), rel=1e-15)
        assert o[0, 0, i, 0] == pytest.approx(
            sum(math.exp(x - m) * (j + 1) for j, x in enumerate(scores)) / ell, rel=1e-14)


def test_worked_example_online_correction():
    """The blockwise recurrence with blocks [90, 80, 70] then [95] applies the
    correction factor exp(90 - 95) to the first block and reproduces the direct
    result."""
    ex = _load_worked_example()
    b1, b2 = ex["block1"], ex["block2"]
    scores = np.array(b1 + b2)
    n = len(scores)
    q = np.ones((1, 1))
    k = scores.reshape(n, 1)
    v = np.eye(n)  # O row = P row, so the whole probability vector is compared
    trace = []
    o_blk, lse_blk = attention_blockwise(q, k, v, 1.0, False, br=1, bc=len(b1), trace=trace)
    assert len(trace) == 2
    assert trace[0][0] == 0.0  # nothing accumulated before the first block
    factor = math.exp(ex["provisional_max"][0] - ex["final_max"][0])
    assert trace[1][0] == pytest.approx(factor, rel=1e-15)
    # direct softmax of the four scores (square oracle problem: every query row is q = 1)
    o_full, lse_full, p_full = oracle.forward(np.ones((1, 1, n, 1)), scores.reshape(1, 1, n, 1),
                                              np.eye(n).reshape(1, 1, n, n), 1.0, False, want_p=True)
    np.testing.assert_allclose(o_blk[0], p_full[0, 0, 0], rtol=1e-14, atol=1e-300)
    assert lse_blk[0] == pytest.approx(lse_full[0, 0, 0], rel=1e-15)
    # and the first block alone, rescaled by the factor, equals its terms under the final max
    first = sum(math.exp(x - ex["provisional_max"][0]) for x in b1) * factor
    assert first == pytest.approx(sum(math.exp(x - ex["final_max"][0]) for x in b1), rel=1e-15)


# -------------------------------------------------------- (a) independent blockwise
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(2, 4, 64, 32), (1, 2, 37, 16)])
def test_blockwise_matches_oracle(shape, causal):
    x = _np_inputs(*shape, seed=1)
    scale = 1.0 / math.sqrt(shape[3])
    o, lse = oracle.forward(x["q"], x["k"], x["v"], scale, causal)
    for br, bc in ((1, 1), (7, 7), (32, 32), (128, 128), (16, 7)):
        ob, lb = attention_blockwise_bhnd(x["q"], x["k"], x["v"], scale, causal, br, bc)
        np.testing.assert_allclose(ob, o, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lb, lse, rtol=1e-12, atol=1e-12)


def test_blockwise_matches_oracle_stress_logits():
    """Logits spanning about +-100 (q, k ~ N(0, 4^2), d = 64, scale 1/8)."""
    x = _np_inputs(1, 2, 96, 64, seed=3, qk_std=4.0)
    o, lse = oracle.forward(x["q"], x["k"], x["v"], 0.125, True)
    s = 0.125 * np.einsum("bhid,bhjd->bhij", x["q"], x["k"])
    assert np.abs(s).max() > 60.0
    ob, lb = attention_blockwise_bhnd(x["q"], x["k"], x["v"], 0.125, True, 32, 32)
    np.testing.assert_allclose(ob, o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lb, lse, rtol=1e-13, atol=1e-12)


# --------------------------------------------------------------- (c) row sums
@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_p_sum_to_one(causal):
    x = _np_inputs(2, 2, 50, 8, seed=2)
    _, _, p = oracle.forward(x["q"], x["k"], x["v"], 0.3, causal, want_p=True)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-14)
    assert (p >= 0).all()
    if causal:
        n = p.shape[-1]
        hidden = np.triu(np.ones((n, n), dtype=bool), k=1)
        assert (p[..., hidden] == 0.0).all()  # no mass on masked keys, exactly
        assert (p[..., ~hidden] > 0.0).all()


# ------------------------------------------------------------- (d) constant V
@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_constant_o(causal):
    x = _np_inputs(1, 3, 40, 16, seed=4)
    c = np.random.default_rng(0).standard_normal(16)
    v = np.broadcast_to(c, x["v"].shape).copy()
    o, _ = oracle.forward(x["q"], x["k"], v, 0.25, causal)
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=1e-14, atol=1e-14)


# --------------------------------------------------------- (e) closed forms
def test_closed_form_single_key():
    """N = 1: O = v0, LSE = scale q0.k0, dQ = dK = 0, dV = dO."""
    rng = np.random.default_rng(5)
    q, k, v, do = (rng.standard_normal((2, 3, 1, 8)) for _ in range(4))
    scale = 0.37
    for causal in (False, True):
        o, lse = oracle.forward(q, k, v, scale, causal)
        np.testing.assert_array_equal(o, v)
        np.testing.assert_allclose(lse, scale * np.einsum("bhnd,bhnd->bhn", q, k), rtol=1e-15)
        dq, dk, dv = oracle.backward(q, k, v, o, do, scale, causal)
        np.testing.assert_allclose(dq, 0.0, atol=1e-15)
        np.testing.assert_allclose(dk, 0.0, atol=1e-15)
        np.testing.assert_array_equal(dv, do)


def test_closed_form_two_keys_d1():
    """d = 1, N = 2: O_i = v0 + (v1 - v0) sigmoid(s q_i (k1 - k0)),
    LSE_i = s q_i k0 + ln(1 + e^{s q_i (k1 - k0)}); causal row 0 sees only key 0."""
    q = np.array([0.7, -1.3]).reshape(1, 1, 2, 1)
    k = np.array([0.4, 2.1]).reshape(1, 1, 2, 1)
    v = np.array([-1.5, 3.0]).reshape(1, 1, 2, 1)
    s = 0.9
    o, lse = oracle.forward(q, k, v, s, False)
    for i in range(2):
        a = s * q[0, 0, i, 0] * (k[0, 0, 1, 0] - k[0, 0, 0, 0])
        sig = 1.0 / (1.0 + math.exp(-a))
        assert o[0, 0, i, 0] == pytest.approx(v[0, 0, 0, 0] + (v[0, 0, 1, 0] - v[0, 0, 0, 0]) * sig, rel=1e-14)
        assert lse[0, 0, i] == pytest.approx(s * q[0, 0, i, 0] * k[0, 0, 0, 0] + math.log1p(math.exp(a)),
                                             rel=1e-14)
    oc, lc = oracle.forward(q, k, v, s, True)
    assert oc[0, 0, 0, 0] == v[0, 0, 0, 0]
    assert lc[0, 0, 0] == pytest.approx(s * q[0, 0, 0, 0] * k[0, 0, 0, 0], rel=1e-15)
    assert oc[0, 0, 1, 0] == pytest.approx(o[0, 0, 1, 0], rel=1e-15)


# ---------------------------------------------------- (f) finite differences
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 2), (3, 2), (5, 3), (4, 1)])
def test_backward_matches_finite_differences(N, d, causal):
    rng = np.random.default_rng(10 * N + d + causal)
    q, k, v, do = (rng.standard_normal((1, 2, N, d)) for _ in range(4))
    scale = 0.8
    o, _ = oracle.forward(q, k, v, scale, causal)
    dq, dk, dv = oracle.backward(q, k, v, o, do, scale, causal)

    def loss(qq, kk, vv):
        oo, _ = oracle.forward(qq, kk, vv, scale, causal, threads=1)
        return float((oo * do).sum())

    h = 1e-6
    for name, grad in (("q", dq), ("k", dk), ("v", dv)):
        base = {"q": q, "k": k, "v": v}
        fd = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            plus = {n: a.copy() for n, a in base.items()}
            minus = {n: a.copy() for n, a in base.items()}
            plus[name][idx] += h
            minus[name][idx] -= h
            fd[idx] = (loss(plus["q"], plus["k"], plus["v"]) - loss(minus["q"], minus["k"], minus["v"])) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8, err_msg=name)


# ------------------------------------------------------------- invariants
def test_causal_row_equals_truncated_problem():
    """Causal row i equals the non-causal answer for the sequence cut after key i,
    and does not change when later keys/values change."""
    x = _np_inputs(1, 2, 33, 16, seed=6)
    scale = 0.25
    o, lse = oracle.forward(x["q"], x["k"], x["v"], scale, True)
    for i in (0, 1, 15, 32):
        sl = slice(0, i + 1)
        ot, lt = oracle.forward(x["q"][:, :, sl], x["k"][:, :, sl], x["v"][:, :, sl], scale, False)
        np.testing.assert_allclose(o[:, :, i], ot[:, :, i], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse[:, :, i], lt[:, :, i], rtol=1e-14)
    k2, v2 = x["k"].copy(), x["v"].copy()
    k2[:, :, 20:] = 7.0
    v2[:, :, 20:] = -3.0
    o2, l2 = oracle.forward(x["q"], k2, v2, scale, True)
    np.testing.assert_array_equal(o2[:, :, :20], o[:, :, :20])
    np.testing.assert_array_equal(l2[:, :, :20], lse[:, :, :20])


def test_key_shift_invariance():
    """K -> K + 1 c^T shifts row i's logits by scale q_i.c: O unchanged, LSE shifted."""
    x = _np_inputs(1, 2, 30, 8, seed=7)
    scale = 0.35
    c = np.random.default_rng(1).standard_normal(8)
    o, lse = oracle.forward(x["q"], x["k"], x["v"], scale, False)
    o2, l2 = oracle.forward(x["q"], x["k"] + c, x["v"], scale, False)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l2, lse + scale * x["q"] @ c, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_column_sums(causal):
    """sum_j dV_j = sum_i dO_i (rows of P sum to 1); sum_j dK_j = 0 (rows of dS sum to 0)."""
    x = _np_inputs(2, 2, 45, 16, seed=8)
    scale = 0.25
    o, _ = oracle.forward(x["q"], x["k"], x["v"], scale, causal)
    dq, dk, dv = oracle.backward(x["q"], x["k"], x["v"], o, x["do"], scale, causal)
    np.testing.assert_allclose(dv.sum(2), x["do"].sum(2), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dk.sum(2), 0.0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_rows_and_cols_match_full(causal):
    """The per-row and per-column entry points (used at sizes where a head
    cannot be materialised) agree with the full materialising pass."""
    x = _np_inputs(2, 3, 70, 16, seed=9)
    scale = 0.25
    o, lse = oracle.forward(x["q"], x["k"], x["v"], scale, causal)
    dq, dk, dv = oracle.backward(x["q"], x["k"], x["v"], o, x["do"], scale, causal)
    of, lf = o.reshape(6, 70, 16), lse.reshape(6, 70)
    bh = np.array([0, 5, 3, 2, 5])
    ri = np.array([0, 69, 17, 40, 1])
    ro, rl, rdq = oracle.rows(x["q"], x["k"], x["v"], x["do"], scale, causal, bh, ri)
    np.testing.assert_allclose(ro, of[bh, ri], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(rl, lf[bh, ri], rtol=1e-14)
    np.testing.assert_allclose(rdq, dq.reshape(6, 70, 16)[bh, ri], rtol=1e-11, atol=1e-13)
    D = (x["do"] * o).sum(-1)
    ck, cv = oracle.cols(x["q"], x["k"], x["v"], x["do"], lse, D, scale, causal, bh, ri)
    np.testing.assert_allclose(ck, dk.reshape(6, 70, 16)[bh, ri], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(cv, dv.reshape(6, 70, 16)[bh, ri], rtol=1e-11, atol=1e-13)


def test_oracle_rejects_bad_arguments():
    x = _np_inputs(1, 1, 4, 4, seed=0)
    with pytest.raises(RuntimeError):
        oracle.rows(x["q"], x["k"], x["v"], None, 1.0, False, np.array([1]), np.array([0]))
    with pytest.raises(RuntimeError):
        oracle.rows(x["q"], x["k"], x["v"], None, 1.0, False, np.array([0]), np.array([4]))


# ------------------------------------------------------- block-sparse mask
def _block_lower(nb):
    return np.tril(np.ones((nb, nb), dtype=np.uint8))[None]


def test_mask_all_ones_is_the_unmasked_definition():
    x = _np_inputs(1, 2, 200, 16, seed=31)
    for causal in (False, True):
        o, l = oracle.forward(x["q"], x["k"], x["v"], 0.3, causal)
        om, lm = oracle.forward(x["q"], x["k"], x["v"], 0.3, causal, block_mask=np.ones((1, 4, 4), np.uint8),
                                blk=64)
        np.testing.assert_array_equal(om, o)
        np.testing.assert_array_equal(lm, l)


def test_lower_block_mask_with_causal_is_causal():
    x = _np_inputs(1, 2, 150, 8, seed=32)
    o, l = oracle.forward(x["q"], x["k"], x["v"], 0.3, True)
    om, lm = oracle.forward(x["q"], x["k"], x["v"], 0.3, True, block_mask=_block_lower(5), blk=32)
    np.testing.assert_array_equal(om, o)
    np.testing.assert_array_equal(lm, l)


def test_block_diagonal_mask_is_independent_blocks():
    """Only diagonal blocks visible = each block of rows attends only to its own
    block of keys, i.e. independent attention problems of length blk."""
    blk, nb = 16, 5
    N = blk * nb - 7  # ragged last block
    x = _np_inputs(1, 3, N, 8, seed=33)
    mask = np.eye(nb, dtype=np.uint8)[None].repeat(3, 0)
    om, lm = oracle.forward(x["q"], x["k"], x["v"], 0.4, False, block_mask=mask, blk=blk)
    for b0 in range(0, N, blk):
        sl = slice(b0, min(b0 + blk, N))
        ob, lb = oracle.forward(x["q"][:, :, sl], x["k"][:, :, sl], x["v"][:, :, sl], 0.4, False)
        np.testing.assert_allclose(om[:, :, sl], ob, rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(lm[:, :, sl], lb, rtol=1e-15)


def test_row_with_no_visible_block_is_zero_with_minus_inf_lse():
    x = _np_inputs(1, 1, 64, 8, seed=34)
    mask = np.ones((1, 4, 4), np.uint8)
    mask[0, 2, :] = 0
    om, lm = oracle.forward(x["q"], x["k"], x["v"], 0.4, False, block_mask=mask, blk=16)
    assert (om[0, 0, 32:48] == 0).all() and np.isneginf(lm[0, 0, 32:48]).all()
    assert np.isfinite(lm[0, 0, :32]).all() and np.isfinite(lm[0, 0, 48:]).all()


@pytest.mark.parametrize("causal", [False, True])
def test_masked_oracle_matches_blockwise_reference(causal):
    blk, N = 32, 150
    nb = (N + blk - 1) // blk
    rng = np.random.default_rng(35)
    mask = (rng.random((2, nb, nb)) < 0.5).astype(np.uint8)
    mask[:, np.arange(nb), np.arange(nb)] = 1
    x = _np_inputs(1, 2, N, 16, seed=36)
    om, lm = oracle.forward(x["q"], x["k"], x["v"], 0.25, causal, block_mask=mask, blk=blk)
    for h in range(2):
        fn = lambda i, j, h=h: mask[h][i // blk, j // blk].astype(bool)  # noqa: E731
        ob, lb = attention_blockwise(x["q"][0, h], x["k"][0, h], x["v"][0, h], 0.25, causal, 16, 24,
                                     mask_fn=fn)
        np.testing.assert_allclose(om[0, h], ob, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lm[0, h], lb, rtol=1e-12, atol=1e-12)


def test_masked_backward_matches_finite_differences():
    rng = np.random.default_rng(37)
    q, k, v, do = (rng.standard_normal((1, 1, 6, 2)) for _ in range(4))
    mask = np.array([[[1, 0, 1], [0, 1, 1], [1, 1, 0]]], dtype=np.uint8)  # blk = 2
    o, _ = oracle.forward(q, k, v, 0.7, False, block_mask=mask, blk=2)
    dq, dk, dv = oracle.backward(q, k, v, o, do, 0.7, False, block_mask=mask, blk=2)

    def loss(qq, kk, vv):
        oo, _ = oracle.forward(qq, kk, vv, 0.7, False, threads=1, block_mask=mask, blk=2)
        return float((oo * do).sum())

    h = 1e-6
    for name, grad in (("q", dq), ("k", dk), ("v", dv)):
        base = {"q": q, "k": k, "v": v}
        fd = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            plus = {n: a.copy() for n, a in base.items()}
            minus = {n: a.copy() for n, a in base.items()}
            plus[name][idx] += h
            minus[name][idx] -= h
            fd[idx] = (loss(plus["q"], plus["k"], plus["v"]) - loss(minus["q"], minus["k"], minus["v"])) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8, err_msg=name)

"""Pins for the oracle's dropout variant (no GPU needed).

The dropout step of the fused kernel (FlashAttention深度攻略 §7, operator
fusion) is read as inverted dropout on the softmax probabilities, with the
keep decisions drawn from Philox4x32-10.  The generator is pinned by its
published known-answer vectors; the draw mapping, the keep rate, the
unbiasedness of the rescaled output, a closed form with uniform scores, and
central finite differences of the dropout forward (which pin the backward,
including the mask in dP and D = rowsum(dO o O)) pin the rest.
"""
import math
import os

import numpy as np
import pytest

import oracle
from io_aware_exact_12_gb300.synth import AttnShape, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _kat_rows():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                w = [int(x, 16) for x in line.split()]
                rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


def _threshold(p):
    return int(math.floor((1.0 - p) * 256.0 + 0.5))


def _np_inputs(B, H, N, d, seed=0):
    t = make_inputs(AttnShape(B, H, N, d), dtype="bf16", seed=seed)
    return {k: v.double().numpy() for k, v in t.items()}


def test_philox_known_answers():
    rows = _kat_rows()
    assert len(rows) == 3
    for ctr, key, want in rows:
        assert oracle.philox4x32_10(ctr, key) == want


def test_keep_mask_follows_the_stated_draw():
    """keep_ij = byte (j mod 4) of word (j mod 16) // 4 of Philox(ctr = (j // 16, i, bh, offset))."""
    p, seed, offset, bh = 0.3, 0x0123456789ABCDEF, 77, 5
    t = _threshold(p)
    keep = oracle.dropout_keep(p, seed, offset, bh, 40, 70)
    rng = np.random.default_rng(0)
    for i, j in zip(rng.integers(0, 40, 200), rng.integers(0, 70, 200)):
        out = oracle.philox4x32_10([j >> 4, i, bh, offset], [seed & 0xFFFFFFFF, seed >> 32])
        byte = (out[(j & 15) >> 2] >> (8 * (j & 3))) & 0xFF
        assert keep[i, j] == int(byte < t), (i, j)


@pytest.mark.parametrize("p", [0.1, 0.5, 0.875])
def test_keep_rate_and_independence(p):
    q = _threshold(p) / 256.0
    keep = oracle.dropout_keep(p, 42, 0, 0, 256, 512).astype(np.float64)
    n = keep.size
    sd = math.sqrt(q * (1 - q) / n)
    assert abs(keep.mean() - q) < 5 * sd
    # neighbouring 16-key groups and neighbouring rows draw independently
    for a, b in ((keep[:, :-16], keep[:, 16:]), (keep[:-1], keep[1:]), (keep[:, :-1], keep[:, 1:])):
        both = (a * b).mean()
        assert abs(both - q * q) < 5 * math.sqrt(q * q * (1 - q * q) / a.size)
    # another head or another offset gives another mask
    for other in (oracle.dropout_keep(p, 42, 0, 1, 256, 512), oracle.dropout_keep(p, 42, 1, 0, 256, 512)):
        agree = (other == keep).mean()
        expect = q * q + (1 - q) * (1 - q)
        assert abs(agree - expect) < 5 * math.sqrt(expect * (1 - expect) / n)


@pytest.mark.parametrize("causal", [False, True])
def test_p_zero_is_the_plain_definition(causal):
    x = _np_inputs(1, 2, 37, 8, seed=3)
    o, lse = oracle.forward(x["q"], x["k"], x["v"], 0.3, causal)
    od, ld = oracle.forward(x["q"], x["k"], x["v"], 0.3, causal, dropout=(0.0, 9, 9))
    np.testing.assert_array_equal(od, o)
    np.testing.assert_array_equal(ld, lse)
    g = oracle.backward(x["q"], x["k"], x["v"], o, x["do"], 0.3, causal)
    gd = oracle.backward(x["q"], x["k"], x["v"], o, x["do"], 0.3, causal, dropout=(0.0, 9, 9))
    for a, b in zip(g, gd):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_scores_closed_form(causal):
    """Q = 0 makes every visible P_ij equal (1/N, or 1/(i+1) causal): with V = 1,
    O_i = (256/t) * (kept keys of row i) * P_ij in every column; LSE = log(#visible)."""
    N, d, p, seed, offset = 45, 4, 0.4, 2024, 3
    t = _threshold(p)
    q = np.zeros((1, 2, N, d))
    k = np.random.default_rng(1).standard_normal((1, 2, N, d))
    v = np.ones((1, 2, N, d))
    o, lse = oracle.forward(q, k, v, 0.5, causal, dropout=(p, seed, offset))
    for h in range(2):
        keep = oracle.dropout_keep(p, seed, offset, h, N, N).astype(np.float64)
        for i in range(N):
            n_vis = i + 1 if causal else N
            kept = keep[i, :n_vis].sum()
            np.testing.assert_allclose(o[0, h, i], (256.0 / t) * kept / n_vis, rtol=1e-13)
            assert lse[0, h, i] == pytest.approx(math.log(n_vis), rel=1e-14)


def test_rescaled_output_is_unbiased():
    """Averaged over independent masks (offsets), O converges to the dropout-free O."""
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((1, 1, 8, 4)) for _ in range(3))
    o_ref, _ = oracle.forward(q, k, v, 0.6, False, threads=1)
    S = 3000
    draws = np.stack([oracle.forward(q, k, v, 0.6, False, threads=1, dropout=(0.5, 11, s))[0] for s in range(S)])
    mean, sd = draws.mean(0), draws.std(0)
    assert np.all(np.abs(mean - o_ref) <= 5 * sd / math.sqrt(S) + 1e-12)
    # and the mean is not the un-rescaled one (which would be (t/256) O)
    assert np.abs(mean - 0.5 * o_ref).max() > 10 * (sd.max() / math.sqrt(S))


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_backward_matches_finite_differences(causal):
    """The mask is fixed by (seed, offset): L = <O, dO> is smooth in q, k, v."""
    rng = np.random.default_rng(40 + causal)
    N, d = 20, 2
    q, k, v, do = (rng.standard_normal((1, 1, N, d)) for _ in range(4))
    drop = (0.3, 123456789, 4)
    o, _ = oracle.forward(q, k, v, 0.9, causal, dropout=drop)
    dq, dk, dv = oracle.backward(q, k, v, o, do, 0.9, causal, dropout=drop)
    keep = oracle.dropout_keep(*drop, 0, N, N)
    assert 0 < keep.sum() < keep.size  # the mask really drops something

    def loss(qq, kk, vv):
        oo, _ = oracle.forward(qq, kk, vv, 0.9, causal, threads=1, dropout=drop)
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


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_rows_and_cols_match_full(causal):
    x = _np_inputs(1, 3, 50, 16, seed=12)
    drop = (0.2, 5, 6)
    o, lse = oracle.forward(x["q"], x["k"], x["v"], 0.25, causal, dropout=drop)
    dq, dk, dv = oracle.backward(x["q"], x["k"], x["v"], o, x["do"], 0.25, causal, dropout=drop)
    bh = np.array([0, 2, 1, 2])
    ri = np.array([0, 49, 17, 33])
    ro, rl, rdq = oracle.rows(x["q"], x["k"], x["v"], x["do"], 0.25, causal, bh, ri, dropout=drop)
    np.testing.assert_allclose(ro, o.reshape(3, 50, 16)[bh, ri], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(rl, lse.reshape(3, 50)[bh, ri], rtol=1e-14)
    np.testing.assert_allclose(rdq, dq.reshape(3, 50, 16)[bh, ri], rtol=1e-11, atol=1e-13)
    D = (x["do"] * o).sum(-1)
    ck, cv = oracle.cols(x["q"], x["k"], x["v"], x["do"], lse, D, 0.25, causal, bh, ri, dropout=drop)
    np.testing.assert_allclose(ck, dk.reshape(3, 50, 16)[bh, ri], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(cv, dv.reshape(3, 50, 16)[bh, ri], rtol=1e-11, atol=1e-13)


def test_dropout_rejects_bad_probability():
    x = _np_inputs(1, 1, 8, 4)
    for p in (1.0, -0.1, float("nan"), 0.999):
        with pytest.raises(RuntimeError):
            oracle.forward(x["q"], x["k"], x["v"], 0.5, False, dropout=(p, 1, 1))


# ---------------------------------------------------------------------------
# Dropout under a block mask.  The keep rule is the one pinned above and does
# not depend on the mask; the mask decides which keys enter the softmax
# (FlashAttention深度攻略 §7 fuses both into the softmax step; 进阶追问
# "Sparse FlashAttention" is the block mask).

def _block_mask(H, nb, density, seed):
    m = (np.random.default_rng(seed).random((H, nb, nb)) < density).astype(np.uint8)
    m[0, 1, :] = 0  # query block 1 of head 0 sees no key
    m[:, :, nb - 1] = 0  # no query block sees the last key block
    m[:, 0, 0] = 1
    return m


@pytest.mark.parametrize("causal", [False, True])
def test_masked_dropout_reads_every_weight(causal):
    """V_j = e_j turns O_i into the weights themselves: key j contributes
    (256/t) keep_ij / n_i when it is visible and nothing otherwise, where n_i
    counts the visible keys of row i (Q = 0 makes their P equal); a row with
    no visible key gives O = 0 and LSE = -inf."""
    N, blk, p, seed, offset = 23, 4, 0.4, 77, 9
    nb = (N + blk - 1) // blk
    H = 2
    mask = _block_mask(H, nb, 0.5, seed=3)
    t = _threshold(p)
    q = np.zeros((1, H, N, N))
    k = np.random.default_rng(2).standard_normal((1, H, N, N))
    v = np.broadcast_to(np.eye(N), (1, H, N, N)).copy()
    o, lse = oracle.forward(q, k, v, 0.3, causal, block_mask=mask, blk=blk, dropout=(p, seed, offset))
    for h in range(H):
        keep = oracle.dropout_keep(p, seed, offset, h, N, N)
        for i in range(N):
            vis = np.array([bool(mask[h, i // blk, j // blk]) and (not causal or j <= i) for j in range(N)])
            n = vis.sum()
            if n == 0:
                assert np.all(o[0, h, i] == 0) and lse[0, h, i] == -np.inf
                continue
            np.testing.assert_allclose(o[0, h, i], (256.0 / t) * (vis & (keep[i] == 1)) / n, rtol=1e-13, atol=0)
            assert lse[0, h, i] == pytest.approx(math.log(n), rel=1e-14)
    assert np.any(lse == -np.inf)  # the empty query block is exercised


@pytest.mark.parametrize("causal", [False, True])
def test_masked_dropout_special_cases(causal):
    """An all-ones mask gives the dropout oracle and p = 0 gives the block-mask
    oracle, bit for bit."""
    x = _np_inputs(1, 2, 37, 8, seed=21)
    nb = (37 + 7) // 8
    ones = np.ones((1, nb, nb), dtype=np.uint8)
    drop = (0.25, 99, 1)
    a = oracle.forward(x["q"], x["k"], x["v"], 0.4, causal, block_mask=ones, blk=8, dropout=drop)
    b = oracle.forward(x["q"], x["k"], x["v"], 0.4, causal, dropout=drop)
    assert all(np.array_equal(u, w) for u, w in zip(a, b))
    ga = oracle.backward(x["q"], x["k"], x["v"], a[0], x["do"], 0.4, causal, block_mask=ones, blk=8, dropout=drop)
    gb = oracle.backward(x["q"], x["k"], x["v"], b[0], x["do"], 0.4, causal, dropout=drop)
    assert all(np.array_equal(u, w) for u, w in zip(ga, gb))
    mask = _block_mask(2, nb, 0.5, seed=8)
    c = oracle.forward(x["q"], x["k"], x["v"], 0.4, causal, block_mask=mask, blk=8, dropout=(0.0, 5, 5))
    e = oracle.forward(x["q"], x["k"], x["v"], 0.4, causal, block_mask=mask, blk=8)
    assert all(np.array_equal(u, w) for u, w in zip(c, e))


@pytest.mark.parametrize("causal", [False, True])
def test_masked_dropout_backward_matches_finite_differences(causal):
    rng = np.random.default_rng(60 + causal)
    N, d, blk = 20, 2, 4
    q, k, v, do = (rng.standard_normal((1, 1, N, d)) for _ in range(4))
    mask = _block_mask(1, N // blk, 0.6, seed=4)
    drop = (0.3, 31337, 2)
    o, _ = oracle.forward(q, k, v, 0.9, causal, block_mask=mask, blk=blk, dropout=drop)
    dq, dk, dv = oracle.backward(q, k, v, o, do, 0.9, causal, block_mask=mask, blk=blk, dropout=drop)
    assert np.all(dk[0, 0, -blk:] == 0) and np.all(dv[0, 0, -blk:] == 0)  # the key block no query sees

    def loss(qq, kk, vv):
        oo, _ = oracle.forward(qq, kk, vv, 0.9, causal, threads=1, block_mask=mask, blk=blk, dropout=drop)
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

"""Block-sparse forward against the float64 oracle with the same block mask
(key j visible to query i iff mask[h][i//128][j//128] != 0, and j <= i if
causal; a row seeing no key has O = 0, LSE = -inf).  Tolerances are the
forward's: max |dO| <= 1e-2 beyond the output type's rounding, max
|dLSE| <= 1e-3; masked structure must hold exactly."""
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


def _random_mask(heads, nb, density, seed, keep_diag=True):
    g = torch.Generator().manual_seed(seed)
    m = (torch.rand((heads, nb, nb), generator=g) < density).to(torch.uint8)
    if keep_diag:
        m[:, torch.arange(nb), torch.arange(nb)] = 1
    return m


def _half_ulp(ref, dtype):
    if dtype == torch.bfloat16:
        return _half_ulp_bf16(ref)
    e = np.floor(np.log2(np.maximum(np.abs(ref), 1e-30)))
    return np.exp2(np.maximum(e, -14) - 11)


def _check(pkg, shape, mask, causal, seed, scale=None, dtype="bf16"):
    x = make_inputs(shape, dtype, seed=seed, with_grad=False)
    scale = 1.0 / math.sqrt(shape.d) if scale is None else scale
    o, lse = pkg.attn_fwd_blocksparse(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), mask.cuda(), scale=scale,
                                      causal=causal)
    assert pkg.sync_status() == 0
    f = lambda t: t.double().numpy()  # noqa: E731
    oo, lo = oracle.forward(f(x["q"]), f(x["k"]), f(x["v"]), scale, causal, block_mask=mask.numpy(), blk=128)
    go, gl = o.double().cpu().numpy(), lse.double().cpu().numpy()
    empty = np.isneginf(lo)
    assert np.array_equal(np.isneginf(gl), empty)            # the same rows see no key
    assert (go[empty] == 0).all()
    err = np.abs(go - oo)
    assert (err - _half_ulp(oo, o.dtype)).max() <= 1e-2, "max|dO| %g" % err.max()
    assert np.abs(gl[~empty] - lo[~empty]).max() <= 1e-3
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1000, 128), (640, 64), (300, 32)])
def test_random_block_masks(pkg, N, d, causal):
    nb = (N + 127) // 128
    _check(pkg, AttnShape(2, 3, N, d), _random_mask(3, nb, 0.4, seed=N + d), causal, seed=N)


def test_shared_mask_and_empty_rows(pkg):
    N, nb = 700, 6
    mask = _random_mask(1, nb, 0.5, seed=3, keep_diag=False)
    mask[0, 2, :] = 0  # query block 2 sees nothing
    mask[0, 0, 0] = 1
    _check(pkg, AttnShape(1, 4, N, 128), mask, False, seed=5)


def test_all_ones_mask_equals_dense_forward_bitwise(pkg):
    shape = AttnShape(1, 2, 900, 128)
    x = make_inputs(shape, "bf16", seed=7, with_grad=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    mask = torch.ones((1, 8, 8), dtype=torch.uint8, device="cuda")
    for causal in (False, True):
        o1, l1 = pkg.attn_fwd(q, k, v, scale=0.1, causal=causal)
        o2, l2 = pkg.attn_fwd_blocksparse(q, k, v, mask, scale=0.1, causal=causal)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_block_diagonal_mask(pkg):
    N, nb = 1024, 8
    mask = torch.eye(nb, dtype=torch.uint8)[None]
    _check(pkg, AttnShape(1, 2, N, 128), mask, False, seed=9)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("N", [1, 127, 129])
def test_small_and_ragged_sequences(pkg, N, d):
    """One and two query tiles, the last one ragged: a CTA's single tile, its
    one- or two-entry key list and the tail mask (forward and backward)."""
    nb = (N + 127) // 128
    for causal in (False, True):
        mask = _random_mask(2, nb, 0.5, seed=N * d + causal)
        _check(pkg, AttnShape(1, 2, N, d), mask, causal, seed=N + d)
        _check_bwd(pkg, AttnShape(1, 2, N, d), mask, causal, seed=N + d + 1)


@pytest.mark.parametrize("d", [64, 128])
def test_all_zero_mask(pkg, d):
    """No key visible anywhere: O = 0 and LSE = -inf in every row, all
    gradients exactly zero, and nothing is loaded."""
    N = 300
    nb = (N + 127) // 128
    x = make_inputs(AttnShape(1, 2, N, d), "bf16", seed=13)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    mask = torch.zeros((1, nb, nb), dtype=torch.uint8, device="cuda")
    o, lse = pkg.attn_fwd_blocksparse(q, k, v, mask, scale=0.1)
    dq, dk, dv = pkg.attn_bwd_blocksparse(q, k, v, o, do, lse, mask, scale=0.1)
    assert pkg.sync_status() == 0
    assert not o.any() and torch.isneginf(lse).all()
    assert not dq.any() and not dk.any() and not dv.any()


def test_sparse_long_sequence_sampled_rows(pkg):
    """N = 8192 with a 25 %-dense mask: sampled rows against the oracle's
    definition on the visible keys of each row (rows of the masked problem)."""
    N, nb, d = 8192, 64, 128
    mask = _random_mask(1, nb, 0.25, seed=11)
    x = make_inputs(AttnShape(1, 2, N, d), "bf16", seed=13, with_grad=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = pkg.attn_fwd_blocksparse(q, k, v, mask.cuda(), scale=1 / math.sqrt(d), causal=False)
    assert pkg.sync_status() == 0
    rng = np.random.default_rng(1)
    for h, i in zip(rng.integers(0, 2, 24), rng.integers(0, N, 24)):
        cols = np.concatenate([np.arange(j * 128, min(N, j * 128 + 128)) for j in range(nb)
                               if mask[0, i // 128, j]])
        qf = x["q"][0, h].double().numpy()
        kf = x["k"][0, h].double().numpy()[cols]
        vf = x["v"][0, h].double().numpy()[cols]
        # the same problem as oracle rows: query i against the visible keys only
        L = len(cols)
        qq = np.zeros((1, 1, L, d))
        qq[0, 0, L - 1] = qf[i]
        ro, rl, _ = oracle.rows(qq, kf[None, None], vf[None, None], None, 1 / math.sqrt(d), False,
                                np.array([0]), np.array([L - 1]))
        go = o[0, h, i].double().cpu().numpy()
        assert (np.abs(go - ro[0]) - _half_ulp_bf16(ro[0])).max() <= 1e-2
        assert abs(lse[0, h, i].item() - rl[0]) <= 1e-3


# ------------------------------------------------------------------ backward
# Gradients against the oracle's masked backward (rel Frobenius <= 2e-2, the
# denominator floored at 1e-3 |dO| where an exact gradient vanishes); key
# tiles no query tile sees must have dK = dV = 0 exactly, and query blocks that
# see no key dQ = 0 exactly.
def _check_bwd(pkg, shape, mask, causal, seed, scale=None, dtype="bf16"):
    x = make_inputs(shape, dtype, seed=seed)
    scale = 1.0 / math.sqrt(shape.d) if scale is None else scale
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    m = mask.cuda()
    o, lse = pkg.attn_fwd_blocksparse(q, k, v, m, scale=scale, causal=causal)
    dq, dk, dv = pkg.attn_bwd_blocksparse(q, k, v, o, do, lse, m, scale=scale, causal=causal)
    assert pkg.sync_status() == 0
    f = lambda t: t.double().cpu().numpy()  # noqa: E731
    oo, _ = oracle.forward(f(x["q"]), f(x["k"]), f(x["v"]), scale, causal, block_mask=mask.numpy(), blk=128)
    ref = oracle.backward(f(x["q"]), f(x["k"]), f(x["v"]), oo, f(x["do"]), scale, causal,
                          block_mask=mask.numpy(), blk=128)
    floor = 1e-3 * float(np.linalg.norm(f(x["do"])))
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        e = float(np.linalg.norm(f(g) - r) / max(np.linalg.norm(r), floor))
        assert e <= 2e-2, "%s rel Frobenius error %g" % (name, e)
    # exact zeros where the mask leaves nothing
    N, nb = shape.N, (shape.N + 127) // 128
    mk = mask.numpy().astype(bool)
    tri = np.tril(np.ones((nb, nb), dtype=bool)) if causal else np.ones((nb, nb), dtype=bool)
    for h in range(shape.H):
        mh = mk[h % mk.shape[0]] & tri
        for j in np.nonzero(~mh.any(axis=0))[0]:      # key tile seen by no query tile
            assert not dk[:, h, j * 128:min(N, j * 128 + 128)].any()
            assert not dv[:, h, j * 128:min(N, j * 128 + 128)].any()
        for i in np.nonzero(~mh.any(axis=1))[0]:      # query block that sees no key
            assert not dq[:, h, i * 128:min(N, i * 128 + 128)].any()
    return dq, dk, dv


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1000, 128), (640, 64), (300, 32)])
def test_backward_random_block_masks(pkg, N, d, causal):
    nb = (N + 127) // 128
    _check_bwd(pkg, AttnShape(2, 3, N, d), _random_mask(3, nb, 0.4, seed=N + d + 1), causal, seed=N + 1)


def test_backward_shared_mask_with_empty_query_block_and_unseen_key_tile(pkg):
    N, nb = 700, 6
    mask = _random_mask(1, nb, 0.5, seed=4, keep_diag=False)
    mask[0, 2, :] = 0  # query block 2 sees nothing
    mask[0, :, 4] = 0  # key tile 4 is seen by no query block
    mask[0, 0, 0] = 1
    for causal in (False, True):
        _check_bwd(pkg, AttnShape(1, 4, N, 128), mask, causal, seed=6)


def test_backward_all_ones_mask_equals_dense(pkg):
    """Same query tiles as the dense backward.  Under the causal mask in the
    same order too: dK and dV bit-identical.  Without it the dense backward
    runs a short grid's key tiles as two CTAs over half the query tiles each
    and adds their fp32 partial dK/dV (the same sums, associated differently),
    so there they agree to the rounding of the bf16 result.  dQ (reduced with
    atomics in any order) to rounding."""
    shape = AttnShape(1, 2, 900, 128)
    x = make_inputs(shape, "bf16", seed=8)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    mask = torch.ones((1, 8, 8), dtype=torch.uint8, device="cuda")
    for causal in (False, True):
        o, lse = pkg.attn_fwd(q, k, v, scale=0.1, causal=causal)
        g1 = pkg.attn_bwd(q, k, v, o, do, lse, scale=0.1, causal=causal)
        g2 = pkg.attn_bwd_blocksparse(q, k, v, o, do, lse, mask, scale=0.1, causal=causal)
        if causal:
            assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
        else:
            for a, b in ((g1[1], g2[1]), (g1[2], g2[2])):
                a, b = a.float(), b.float()
                ulp = torch.exp2(torch.floor(torch.log2(b.abs().clamp_min(1e-30))) - 7)  # one bf16 ulp at b
                assert ((a - b).abs() <= ulp + 1e-6 * b.abs().max()).all()
        assert (g1[0].float() - g2[0].float()).abs().max().item() <= 1e-2 * g1[0].float().abs().max().item()


def test_sparse_beyond_512_tiles(pkg):
    """N = 66176 (517 key tiles, past the former 512-tile limit), a 4 %-dense
    mask: sampled forward rows against the oracle on each row's visible keys;
    the backward runs, and key tiles no query tile sees get dK = dV = 0."""
    N, d = 66176, 64
    nb = (N + 127) // 128
    mask = _random_mask(1, nb, 0.04, seed=31)
    mask[0, :, 515] = 0                        # one key tile nobody sees
    x = make_inputs(AttnShape(1, 1, N, d), "bf16", seed=32)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    m = mask.cuda()
    o, lse = pkg.attn_fwd_blocksparse(q, k, v, m, scale=1 / math.sqrt(d), causal=False)
    assert pkg.sync_status() == 0
    rng = np.random.default_rng(3)
    for i in list(rng.integers(0, N, 12)) + [N - 1]:
        cols = np.concatenate([np.arange(j * 128, min(N, j * 128 + 128)) for j in range(nb) if mask[0, i // 128, j]])
        L = len(cols)
        qq = np.zeros((1, 1, L, d))
        qq[0, 0, L - 1] = x["q"][0, 0, i].double().numpy()
        ro, rl, _ = oracle.rows(qq, x["k"][0, 0].double().numpy()[cols][None, None],
                                x["v"][0, 0].double().numpy()[cols][None, None], None, 1 / math.sqrt(d), False,
                                np.array([0]), np.array([L - 1]))
        go = o[0, 0, i].double().cpu().numpy()
        assert (np.abs(go - ro[0]) - _half_ulp_bf16(ro[0])).max() <= 1e-2
        assert abs(lse[0, 0, i].item() - rl[0]) <= 1e-3
    dq, dk, dv = pkg.attn_bwd_blocksparse(q, k, v, o, do, lse, m, scale=1 / math.sqrt(d), causal=False)
    assert pkg.sync_status() == 0
    assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()
    assert not dk[0, 0, 515 * 128:516 * 128].any() and not dv[0, 0, 515 * 128:516 * 128].any()
    assert dk[0, 0, 514 * 128:515 * 128].any() or not mask[0, :, 514].any()


def test_backward_sparse_longer_sequence(pkg):
    """N = 4096, 25 %-dense per-head masks, causal and not, against the full oracle."""
    N, nb = 4096, 32
    for causal in (False, True):
        _check_bwd(pkg, AttnShape(1, 2, N, 128), _random_mask(2, nb, 0.25, seed=21 + causal), causal, seed=22)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1000, 128), (300, 32)])
def test_fp16_random_block_masks_forward_and_backward(pkg, N, d, causal):
    """The fp16 twins of the block-sparse forward and backward."""
    nb = (N + 127) // 128
    mask = _random_mask(3, nb, 0.4, seed=N + d + 7)
    o, _ = _check(pkg, AttnShape(2, 3, N, d), mask, causal, seed=N + 3, dtype="fp16")
    assert o.dtype == torch.float16
    dq, dk, dv = _check_bwd(pkg, AttnShape(2, 3, N, d), mask, causal, seed=N + 4, dtype="fp16")
    assert dq.dtype == torch.float16

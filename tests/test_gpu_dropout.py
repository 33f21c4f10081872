"""GPU parity of the dropout forward and backward against the float64 oracle.

The keep decisions are integer work and are checked bit-exactly: with Q = 0
every visible probability is equal, so choosing V (forward) or dO (backward)
as scaled unit vectors makes each output element an integer count of kept
entries that can be read back exactly and compared with the oracle's
keep_ij for every (i, j) of a head.  O, LSE and dQ/dK/dV are compared with
the tolerances of the plain path (max |dO| <= 1e-2 beyond the output's own
rounding, max |dLSE| <= 1e-3, relative Frobenius error <= 2e-2), in full on
small and ragged shapes and on sampled rows and key columns at B=2, H=16,
N=8192, d=128.

The backward is given O in bf16, so its D_i = sum_k dO_ik O_ik carries the
rounding of O: |D_kernel - D| <= delta_i = sum_k |dO_ik| ulp(O_ik).  That
error enters dS_ij as P_ij delta_i, hence dQ_i by up to scale delta_i
sum_j P_ij |K_j| and dK_j by up to scale sum_i P_ij delta_i |Q_i|.  Without
dropout O = V exactly at N = 1 and the term vanishes; with dropout it does
not, and there the exact dQ and dK are zero.  The full comparisons allow this
term (computed from the oracle's own O and P) on top of the 2e-2 bound.
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


def f64(t):
    return t.detach().double().cpu().numpy()


def half_ulp_bf16(ref):
    e = np.floor(np.log2(np.maximum(np.abs(ref), 1e-30)))
    return np.exp2(e - 8)


def half_ulp(ref, dtype):
    """Half an ulp of the output format (bf16 or fp16) at the exact value."""
    if dtype == torch.bfloat16:
        return half_ulp_bf16(ref)
    e = np.floor(np.log2(np.maximum(np.abs(ref), 1e-30)))
    return np.exp2(np.maximum(e, -14) - 11)


def rel_fro(a, b, floor=1e-30):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), floor))


def threshold(p):
    return int(math.floor((1.0 - float(np.float32(p))) * 256.0 + 0.5))


def run(x, scale, causal, drop):
    pkg = _pkg()
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    p, seed, off = drop
    o, lse = pkg.attn_fwd_dropout(q, k, v, p, seed, off, scale=scale, causal=causal)
    grads = pkg.attn_bwd_dropout(q, k, v, o, do, lse, p, seed, off, scale=scale, causal=causal)
    assert pkg.sync_status() == 0
    return o, lse, grads


def check_full(x, scale, causal, drop, o, lse, grads, block_mask=None):
    d32 = (float(np.float32(drop[0])), drop[1], drop[2])
    q, k, v, do = (f64(x[n]) for n in ("q", "k", "v", "do"))
    bm = None if block_mask is None else block_mask.cpu().numpy()
    oo, lo, P = oracle.forward(q, k, v, scale, causal, want_p=True, block_mask=bm, dropout=d32)
    err = np.abs(f64(o) - oo)
    assert (err - half_ulp(oo, o.dtype)).max() <= TOL_O, "max|dO| %g" % err.max()
    empty = np.isneginf(lo)  # rows that see no key (block mask): LSE = -inf, O = 0
    assert np.array_equal(np.isneginf(f64(lse)), empty)
    assert np.abs(f64(lse)[~empty] - lo[~empty]).max() <= TOL_LSE
    ref = oracle.backward(q, k, v, oo, do, scale, causal, block_mask=bm, dropout=d32)
    floor = 1e-3 * float(np.linalg.norm(do))
    delta = (np.abs(do) * 2 * half_ulp(oo, o.dtype)).sum(-1)  # [B, H, N]
    extra = {"dq": abs(scale) * delta[..., None] * (P @ np.abs(k)),
             "dk": abs(scale) * np.einsum("bhij,bhi,bhic->bhjc", P, delta, np.abs(q)),
             "dv": np.zeros_like(do)}
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        err = float(np.linalg.norm(f64(g) - r))
        allowed = TOL_GRAD * max(float(np.linalg.norm(r)), floor) + float(np.linalg.norm(extra[name]))
        assert err <= allowed, "%s error %g > %g (|ref| %g)" % (name, err, allowed, np.linalg.norm(r))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("p", [0.1, 0.5])
def test_small_full(causal, p):
    x = make_inputs(AttnShape(2, 4, 64, 32), "bf16", seed=21)
    drop = (p, 0x1234_5678_9ABC_DEF0, 3)
    o, lse, grads = run(x, 1 / math.sqrt(32), causal, drop)
    check_full(x, 1 / math.sqrt(32), causal, drop, o, lse, grads)


@pytest.mark.parametrize("N", [1, 17, 127, 129, 300])
@pytest.mark.parametrize("d", [32, 64, 128])
def test_ragged_full(N, d):
    x = make_inputs(AttnShape(1, 3, N, d), "bf16", seed=N + d)
    for causal in (False, True):
        drop = (0.2, 77 + N, d)
        o, lse, grads = run(x, 1 / math.sqrt(d), causal, drop)
        check_full(x, 1 / math.sqrt(d), causal, drop, o, lse, grads)


@pytest.mark.parametrize("d", [32, 64, 128])
def test_fp16_full(d):
    """The fp16 twins: the same keep decisions (the draws do not depend on the
    input type), parity with the oracle on fp16-rounded inputs."""
    x = make_inputs(AttnShape(2, 3, 300, d), "fp16", seed=40 + d)
    for causal in (False, True):
        drop = (0.15, 0xC0FFEE + d, 5)
        o, lse, grads = run(x, 1 / math.sqrt(d), causal, drop)
        assert o.dtype == torch.float16 and grads[0].dtype == torch.float16
        check_full(x, 1 / math.sqrt(d), causal, drop, o, lse, grads)


def _decode_counts(val, denom, t):
    """val = (256/t) * count / denom for integer counts: read the counts back."""
    c = np.rint(val * denom * t / 256.0)
    assert np.abs(val * denom * t / 256.0 - c).max() < 0.1
    return c.astype(np.int64)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_keep_mask_is_bit_exact(causal):
    """Q = 0, V_j = 2^(j // 128) e_(j mod 128): O_ic counts the kept keys
    c, c + 128, ... of row i in binary; every keep_ij of 3 heads x 512 x 512."""
    B, H, N, d = 1, 3, 512, 128
    p, seed, off = 0.3, 0xDEADBEEF_00C0FFEE, 11
    t = threshold(p)
    q = torch.zeros(B, H, N, d, dtype=torch.bfloat16, device="cuda")
    k = make_inputs(AttnShape(B, H, N, d), "bf16", seed=5)["k"].cuda()
    j = torch.arange(N)
    v = torch.zeros(N, d)
    v[j, j % 128] = torch.exp2((j // 128).float())
    v = v.expand(B, H, N, d).contiguous().to(torch.bfloat16).cuda()
    pkg = _pkg()
    o, lse = pkg.attn_fwd_dropout(q, k, v, p, seed, off, scale=0.1, causal=causal)
    assert pkg.sync_status() == 0
    o = f64(o)
    i = np.arange(N)
    n_vis = (i + 1) if causal else np.full(N, N)
    np.testing.assert_allclose(f64(lse)[0], np.log(n_vis)[None, :].repeat(H, 0), atol=1e-5)
    for h in range(H):
        cnt = _decode_counts(o[0, h], n_vis[:, None].astype(np.float64), t)  # [N, 128]
        keep = oracle.dropout_keep(float(np.float32(p)), seed, off, h, N, N).astype(np.int64)
        if causal:
            keep = np.tril(keep)
        want = sum(keep[:, 128 * m:128 * (m + 1)] << m for m in range(4))
        np.testing.assert_array_equal(cnt, want)


def test_backward_keep_mask_is_bit_exact():
    """Q = 0 (P = 1/N), dO_i = 2^(i // 128) e_(i mod 128): dV_jc counts the
    kept queries c, c + 128, ... of key j in binary."""
    B, H, N, d = 1, 2, 512, 128
    p, seed, off = 0.6, 987654321, 2
    t = threshold(p)
    q = torch.zeros(B, H, N, d, dtype=torch.bfloat16, device="cuda")
    k = make_inputs(AttnShape(B, H, N, d), "bf16", seed=6)["k"].cuda()
    v = make_inputs(AttnShape(B, H, N, d), "bf16", seed=7)["v"].cuda()
    i = torch.arange(N)
    do = torch.zeros(N, d)
    do[i, i % 128] = torch.exp2((i // 128).float())
    do = do.expand(B, H, N, d).contiguous().to(torch.bfloat16).cuda()
    pkg = _pkg()
    o, lse = pkg.attn_fwd_dropout(q, k, v, p, seed, off, scale=0.1, causal=False)
    dq, dk, dv = pkg.attn_bwd_dropout(q, k, v, o, do, lse, p, seed, off, scale=0.1, causal=False)
    assert pkg.sync_status() == 0
    dv = f64(dv)
    for h in range(H):
        cnt = _decode_counts(dv[0, h], float(N), t)  # [N keys, 128]
        keep = oracle.dropout_keep(float(np.float32(p)), seed, off, h, N, N).astype(np.int64)  # [query, key]
        kt = keep.T
        want = sum(kt[:, 128 * m:128 * (m + 1)] << m for m in range(4))
        np.testing.assert_array_equal(cnt, want)


@pytest.mark.parametrize("causal", [False, True])
def test_long_sequence_sampled(causal):
    """B=2 H=16 N=8192 d=128, p = 0.1: sampled rows (O, LSE, dQ) and key columns (dK, dV)."""
    shape = AttnShape(2, 16, 8192, 128)
    x = make_inputs(shape, "bf16", seed=4)
    s = 1 / math.sqrt(128)
    drop = (0.1, 2024, 7)
    d32 = (float(np.float32(drop[0])), drop[1], drop[2])
    o, lse, grads = run(x, s, causal, drop)
    q, k, v, do = (f64(x[n]) for n in ("q", "k", "v", "do"))
    N, d = shape.N, shape.d
    bh, ri = sample_rows(shape, 256, seed=12)
    ro, rl, rdq = oracle.rows(q, k, v, do, s, causal, bh, ri, dropout=d32)
    go = f64(o).reshape(-1, N, d)[bh, ri]
    err = np.abs(go - ro)
    assert (err - half_ulp_bf16(ro)).max() <= TOL_O
    assert np.abs(f64(lse).reshape(-1, N)[bh, ri] - rl).max() <= TOL_LSE
    assert rel_fro(f64(grads[0]).reshape(-1, N, d)[bh, ri], rdq) <= TOL_GRAD
    h = 31
    fo, fl, _ = oracle.rows(q, k, v, None, s, causal, np.full(N, h), np.arange(N), dropout=d32)
    lse_all = np.zeros((shape.B * shape.H, N))
    D_all = np.zeros_like(lse_all)
    lse_all[h] = fl
    D_all[h] = (do.reshape(-1, N, d)[h] * fo).sum(-1)
    cols = np.random.default_rng(3).choice(N, size=48, replace=False)
    cols[:2] = [0, N - 1]
    dk_ref, dv_ref = oracle.cols(q, k, v, do, lse_all.reshape(2, 16, N), D_all.reshape(2, 16, N), s, causal,
                                 np.full(48, h), cols, dropout=d32)
    assert rel_fro(f64(grads[1]).reshape(-1, N, d)[h, cols], dk_ref) <= TOL_GRAD
    assert rel_fro(f64(grads[2]).reshape(-1, N, d)[h, cols], dv_ref) <= TOL_GRAD


def test_tiny_probability_is_the_plain_path_and_draws_are_reproducible():
    pkg = _pkg()
    x = make_inputs(AttnShape(1, 2, 200, 64), "bf16", seed=8)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o0, l0 = pkg.attn_fwd(q, k, v, scale=0.125)
    o1, l1 = pkg.attn_fwd_dropout(q, k, v, 0.001, 5, 0, scale=0.125)  # t = 256: nothing dropped
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    a, _ = pkg.attn_fwd_dropout(q, k, v, 0.25, 5, 0, scale=0.125)
    b, _ = pkg.attn_fwd_dropout(q, k, v, 0.25, 5, 0, scale=0.125)
    c, _ = pkg.attn_fwd_dropout(q, k, v, 0.25, 5, 1, scale=0.125)
    assert torch.equal(a, b) and not torch.equal(a, c)
    assert pkg.sync_status() == 0


def test_bad_probability_is_rejected():
    pkg = _pkg()
    x = make_inputs(AttnShape(1, 1, 16, 64), "bf16", seed=9)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    for p in (1.0, -0.5, float("nan"), 0.999):
        with pytest.raises(pkg.AttnError):
            pkg.attn_fwd_dropout(q, k, v, p, 1, 0)
    with pytest.raises(TypeError):  # bf16 or fp16 only
        pkg.attn_fwd_dropout(q.float(), k.float(), v.float(), 0.1, 1, 0)
    with pytest.raises(TypeError):  # one type for all inputs
        pkg.attn_fwd_dropout(q, k.half(), v, 0.1, 1, 0)


# ---------------------------------------------------------------------------
# Dropout under a block mask (attn_fwd_blocksparse_dropout and its backward):
# the keep decisions are those above, applied to the keys the mask leaves
# visible; skipped key tiles shift which key tile a CTA visits next, so the
# draws must follow the tile actually visited.

def run_sparse(x, mask, scale, causal, drop):
    pkg = _pkg()
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    m = mask.cuda()
    p, seed, off = drop
    o, lse = pkg.attn_fwd_blocksparse_dropout(q, k, v, m, p, seed, off, scale=scale, causal=causal)
    grads = pkg.attn_bwd_blocksparse_dropout(q, k, v, o, do, lse, m, p, seed, off, scale=scale, causal=causal)
    assert pkg.sync_status() == 0
    return o, lse, grads


def _sparse_mask(heads, nb, density, seed):
    g = torch.Generator().manual_seed(seed)
    m = (torch.rand((heads, nb, nb), generator=g) < density).to(torch.uint8)
    m[:, torch.arange(nb), torch.arange(nb)] = 1
    m[0, 1, :] = 0  # query block 1 of head 0 sees no key
    m[:, :, nb - 1] = 0  # no query block sees the last key block
    return m


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_blocksparse_full(d, causal):
    N = 1000  # 8 tiles, the last one ragged
    x = make_inputs(AttnShape(1, 3, N, d), "bf16", seed=90 + d)
    mask = _sparse_mask(3, 8, 0.4, seed=d + causal)
    drop = (0.5, 0x5EED_0000_0000_0001 + d, 7)
    o, lse, grads = run_sparse(x, mask, 1 / math.sqrt(d), causal, drop)
    check_full(x, 1 / math.sqrt(d), causal, drop, o, lse, grads, block_mask=mask)


def test_blocksparse_fp16_full():
    x = make_inputs(AttnShape(2, 2, 600, 64), "fp16", seed=97)
    mask = _sparse_mask(1, 5, 0.5, seed=3)
    for causal in (False, True):
        drop = (0.2, 4242, causal)
        o, lse, grads = run_sparse(x, mask, 0.125, causal, drop)
        assert o.dtype == torch.float16 and grads[0].dtype == torch.float16
        check_full(x, 0.125, causal, drop, o, lse, grads, block_mask=mask)


def _two_per_row_mask(H, nb, seed):
    """Every query block sees exactly two key blocks (so every row has the
    same 256 visible keys), chosen at random per head."""
    g = np.random.default_rng(seed)
    m = np.zeros((H, nb, nb), dtype=np.uint8)
    for h in range(H):
        for r in range(nb):
            m[h, r, g.choice(nb, 2, replace=False)] = 1
    return torch.from_numpy(m)


def test_blocksparse_keep_mask_is_bit_exact():
    """The forward and backward readbacks above under a block mask with two
    key blocks per query block: O_ic = (256/t)/256 sum_m keep_i,128m+c
    vis 2^m and dV_jc = (256/t)/256 sum_m keep_128m+c,j vis 2^m, so every
    keep decision of a visible pair is read back as a bit."""
    B, H, N, d = 1, 3, 512, 128
    nb = N // 128
    p, seed, off = 0.45, 0xABCDEF_12345678, 21
    t = threshold(p)
    mask = _two_per_row_mask(H, nb, seed=12)
    mnp = mask.numpy().astype(np.int64)
    q = torch.zeros(B, H, N, d, dtype=torch.bfloat16, device="cuda")
    k = make_inputs(AttnShape(B, H, N, d), "bf16", seed=15)["k"].cuda()
    j = torch.arange(N)
    unit = torch.zeros(N, d)
    unit[j, j % 128] = torch.exp2((j // 128).float())
    unit = unit.expand(B, H, N, d).contiguous().to(torch.bfloat16).cuda()
    pkg = _pkg()
    m = mask.cuda()
    o, lse = pkg.attn_fwd_blocksparse_dropout(q, k, unit, m, p, seed, off, scale=0.1)
    _, _, dv = pkg.attn_bwd_blocksparse_dropout(q, k, unit, o, unit, lse, m, p, seed, off, scale=0.1)
    assert pkg.sync_status() == 0
    np.testing.assert_allclose(f64(lse)[0], math.log(256.0), atol=1e-5)
    o, dv = f64(o), f64(dv)
    for h in range(H):
        keep = oracle.dropout_keep(float(np.float32(p)), seed, off, h, N, N).astype(np.int64)  # [query, key]
        vis = np.kron(mnp[h], np.ones((128, 128), dtype=np.int64))
        kv = keep * vis
        cnt = _decode_counts(o[0, h], 256.0, t)  # [N queries, 128]
        np.testing.assert_array_equal(cnt, sum(kv[:, 128 * b:128 * (b + 1)] << b for b in range(nb)))
        cnt = _decode_counts(dv[0, h], 256.0, t)  # [N keys, 128]
        kt = kv.T
        np.testing.assert_array_equal(cnt, sum(kt[:, 128 * b:128 * (b + 1)] << b for b in range(nb)))


def test_blocksparse_all_ones_equals_dropout_kernels():
    """With every tile enabled the block-sparse kernels visit the tiles of the
    dense ones in the same order: the forward is bit-identical; the backward
    as in the block-sparse tests without dropout (dK, dV bit-identical under
    the causal mask, to one bf16 ulp without it; dQ to rounding)."""
    x = make_inputs(AttnShape(1, 2, 900, 128), "bf16", seed=31)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    mask = torch.ones((1, 8, 8), dtype=torch.uint8, device="cuda")
    pkg = _pkg()
    drop = (0.25, 555, 3)
    for causal in (False, True):
        o1, l1 = pkg.attn_fwd_dropout(q, k, v, *drop, scale=0.1, causal=causal)
        o2, l2 = pkg.attn_fwd_blocksparse_dropout(q, k, v, mask, *drop, scale=0.1, causal=causal)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
        g1 = pkg.attn_bwd_dropout(q, k, v, o1, do, l1, *drop, scale=0.1, causal=causal)
        g2 = pkg.attn_bwd_blocksparse_dropout(q, k, v, o1, do, l1, mask, *drop, scale=0.1, causal=causal)
        if causal:
            assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
        else:
            for a, b in ((g1[1], g2[1]), (g1[2], g2[2])):
                a, b = a.float(), b.float()
                ulp = torch.exp2(torch.floor(torch.log2(b.abs().clamp_min(1e-30))) - 7)
                assert ((a - b).abs() <= ulp + 1e-6 * b.abs().max()).all()
        assert (g1[0].float() - g2[0].float()).abs().max().item() <= 1e-2 * g1[0].float().abs().max().item()
    assert pkg.sync_status() == 0

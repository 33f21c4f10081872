"""Independent blockwise online-softmax reference (NumPy, float64).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  This is a second,
separately written statement of the forward pass, used to cross-check the
materialising C oracle.  It follows the running-statistics recurrence of
FlashAttention (PKM page) §"三招" 2 Online Softmax; the same recurrence is
told in words in "Flash Attention 到底做了什么？" (the section on why blockwise
softmax equals the whole-row softmax) and derived in FlashAttention深度攻略 §4.
The printed form of the recurrence is scrambled by text extraction; it is
read as

    m_j   = max(m_{j-1}, rowmax(S_j))
    Pt_j  = exp(S_j - m_j)
    l_j   = exp(m_{j-1} - m_j) l_{j-1} + rowsum(Pt_j)
    O_j   = diag(exp(m_{j-1} - m_j)) O_{j-1} + Pt_j V_j
    O     = diag(l_last)^-1 O_last                  (final division, same section)

with query blocks of ``br`` rows as the outer loop and key/value blocks of
``bc`` rows as the inner loop (the order of the live-coding module of
FlashAttention深度攻略), and the causal mask applied with global indices (key
j hidden from query i iff j > i).  The module printed there masks each block with a block-local
upper-triangular mask and broadcasts P against V without a sum; neither is
followed: both contradict the plain definition the same page compares it to.
"""
from __future__ import annotations

import numpy as np


def attention_blockwise(q, k, v, scale, causal, br=32, bc=32, trace=None, mask_fn=None):
    """q: [N, d], k, v: [Nk, d] float64 for one head.  Returns (o [N, d], lse [N]).

    ``mask_fn(i, j)``: optional visibility rule on index arrays (True = key j
    visible to query i), applied on top of the causal rule.
    ``trace``: optional list; for each (query block, key block) step the
    rescale factors exp(m_{j-1} - m_j) of that step are appended, so a test
    can observe the correction the pages describe.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, d = q.shape
    nk = k.shape[0]
    o_out = np.zeros((n, v.shape[1]))
    lse_out = np.zeros(n)
    for r0 in range(0, n, br):
        r1 = min(r0 + br, n)
        qi = q[r0:r1]
        m = np.full(r1 - r0, -np.inf)
        l = np.zeros(r1 - r0)
        acc = np.zeros((r1 - r0, v.shape[1]))
        rows = np.arange(r0, r1)[:, None]
        for c0 in range(0, nk, bc):
            c1 = min(c0 + bc, nk)
            if causal and c0 > r1 - 1:
                break  # every key of this block lies after every query of the row block
            s = scale * (qi @ k[c0:c1].T)
            if causal:
                cols = np.arange(c0, c1)[None, :]
                s = np.where(cols > rows, -np.inf, s)
            if mask_fn is not None:  # mask_fn(i, j) -> bool arrays: is key j visible to query i
                s = np.where(mask_fn(rows, np.arange(c0, c1)[None, :]), s, -np.inf)
            m_new = np.maximum(m, s.max(axis=1))
            # rows whose keys so far are all hidden keep m = -inf; guard exp(-inf - -inf)
            safe = np.where(np.isfinite(m_new), m_new, 0.0)
            corr = np.where(np.isfinite(m), np.exp(m - safe), 0.0)
            pt = np.exp(s - safe[:, None])
            l = corr * l + pt.sum(axis=1)
            acc = corr[:, None] * acc + pt @ v[c0:c1]
            if trace is not None:
                trace.append(corr.copy())
            m = m_new
        seen = l > 0  # rows that saw no key at all: O = 0, LSE = -inf
        o_out[r0:r1] = np.where(seen[:, None], acc / np.where(seen, l, 1.0)[:, None], 0.0)
        lse_out[r0:r1] = np.where(seen, m + np.log(np.where(seen, l, 1.0)), -np.inf)
    return o_out, lse_out


def attention_blockwise_bhnd(q, k, v, scale, causal, br=32, bc=32):
    """[B, H, N, d] wrapper: runs every head independently."""
    q = np.asarray(q, dtype=np.float64)
    B, H, N, d = q.shape
    o = np.zeros((B, H, N, v.shape[-1]))
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = attention_blockwise(q[b, h], k[b, h], v[b, h], scale, causal, br, bc)
    return o, lse

"""Seeded synthetic inputs for attention, shared by the CUDA path's tests and
bench and by the CPU oracle's tests.

This module holds none of the method's arithmetic: it only draws Gaussian
numbers from a seeded torch generator and rounds them (round-to-nearest-even)
to the storage dtype, so that the oracle (which upcasts the rounded values
exactly to float64) and the CUDA kernels see bit-identical inputs.

Recipe: every tensor is [B, H, N, d] contiguous; values are i.i.d. N(0, 1)
drawn in float32 in the order q, k, v, dO from ``torch.Generator`` seeded with
``seed``, optionally multiplied by ``qk_std`` for q and k (the logit-range
stress variant uses qk_std = 4, so logits at scale 1/8, d = 64 have standard
deviation 16 and span roughly +-100), then rounded to bf16 or fp16.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

DTYPES = {"bf16": torch.bfloat16, "f16": torch.float16, "fp16": torch.float16}


@dataclass(frozen=True)
class AttnShape:
    B: int
    H: int
    N: int
    d: int

    @property
    def numel(self) -> int:
        return self.B * self.H * self.N * self.d


def make_inputs(shape: AttnShape, dtype: str = "bf16", seed: int = 0, qk_std: float = 1.0,
                with_grad: bool = True, device: str = "cpu"):
    """Return dict(q, k, v[, do]) of [B, H, N, d] tensors in ``dtype``.

    The draw happens on the CPU generator (so it is identical on every
    machine) and is then moved to ``device``.
    """
    td = DTYPES[dtype]
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    dims = (shape.B, shape.H, shape.N, shape.d)
    out = {}
    for name in ("q", "k", "v", "do") if with_grad else ("q", "k", "v"):
        x = torch.randn(dims, generator=g, dtype=torch.float32)
        if name in ("q", "k") and qk_std != 1.0:
            x = x * qk_std
        out[name] = x.to(td).contiguous().to(device)
    return out


def sample_rows(shape: AttnShape, count: int, seed: int = 1234):
    """Seeded (flattened head, row) pairs: a sample of ``count`` query rows that
    always includes the first and last rows of the first and last heads."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    BH = shape.B * shape.H
    bh = torch.randint(0, BH, (count,), generator=g)
    rows = torch.randint(0, shape.N, (count,), generator=g)
    fixed_bh = torch.tensor([0, 0, BH - 1, BH - 1])
    fixed_rows = torch.tensor([0, shape.N - 1, 0, shape.N - 1])
    bh = torch.cat([fixed_bh, bh])[:max(count, 4)]
    rows = torch.cat([fixed_rows, rows])[:max(count, 4)]
    return bh.numpy(), rows.numpy()


E4M3_MAX = 448.0


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor e4m3 quantisation for FP8 inputs: descale = amax / 448 and
    x8 = round-to-nearest-even(x / descale) in float8_e4m3fn, so that
    descale * x8 approximates x.  Returns (x8 as uint8 bytes, descale).  The
    real input both sides use is exactly descale * float(x8)."""
    amax = float(x.abs().max())
    descale = amax / E4M3_MAX if amax > 0 else 1.0
    x8 = (x.float() / descale).to(torch.float8_e4m3fn)
    return x8.view(torch.uint8).contiguous(), descale


def make_inputs_fp8(shape: AttnShape, seed: int = 0, qk_std: float = 1.0):
    """The make_inputs draws (fp32, same order and seed), each tensor then
    quantised per tensor to e4m3.  Returns dict name -> (uint8 bytes, descale)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    dims = (shape.B, shape.H, shape.N, shape.d)
    out = {}
    for name in ("q", "k", "v"):
        x = torch.randn(dims, generator=g, dtype=torch.float32)
        if name in ("q", "k") and qk_std != 1.0:
            x = x * qk_std
        out[name] = quantize_e4m3(x)
    return out


def dequantize_e4m3(x8: torch.Tensor, descale: float) -> torch.Tensor:
    """float64 real values descale * e4m3 (exact)."""
    return x8.view(torch.float8_e4m3fn).double() * descale

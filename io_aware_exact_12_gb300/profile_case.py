"""Runs one attention op a fixed number of times on synthetic inputs, for
capturing it under a profiler (ncu).  Warm-up launches come first, so a
capture can skip them with ``-s``.

  python -m io_aware_exact_12_gb300.profile_case --op fwd --B 2 --H 16 --N 8192 --d 128 --launches 2
  python -m io_aware_exact_12_gb300.profile_case --op bwd ...   (one attn_bwd = 3 launches)
  python -m io_aware_exact_12_gb300.profile_case --op naive ... (materialising 3-step
      torch comparator: S = QK^T, P = softmax(S), O = PV, to measure its DRAM bytes)
  --op fwd_dropout / bwd_dropout: the dropout entries with p = 0.1
  --op decode: one query token per head against an N-token cache (B, H, N, d)
  --op fwd_blocksparse / bwd_blocksparse: a seeded random 25 %-dense per-head
      block mask (diagonal on), as in bench.py
  --op fwd_fp8: the e4m3 forward (d = 128) on per-tensor-quantised inputs
"""
from __future__ import annotations

import argparse
import math

import torch


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", choices=["fwd", "bwd", "naive", "fwd_dropout", "bwd_dropout", "decode",
                                     "fwd_blocksparse", "bwd_blocksparse", "fwd_fp8"], default="fwd")
    ap.add_argument("--B", type=int, default=2)
    ap.add_argument("--H", type=int, default=16)
    ap.add_argument("--N", type=int, default=8192)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--dtype", default="bf16")
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--launches", type=int, default=2)
    a = ap.parse_args(argv)

    import io_aware_exact_12_gb300 as attn
    from io_aware_exact_12_gb300.synth import AttnShape, make_inputs
    x = make_inputs(AttnShape(a.B, a.H, a.N, a.d), a.dtype, seed=4, device="cuda")
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    scale = 1.0 / math.sqrt(a.d)
    o, lse = attn.attn_fwd(q, k, v, scale=scale, causal=a.causal)
    if a.op.endswith("dropout"):
        o, lse = attn.attn_fwd_dropout(q, k, v, 0.1, 1234, 0, scale=scale, causal=a.causal)
    q1 = q[:, :, 0].contiguous()
    if a.op == "fwd_fp8":
        from io_aware_exact_12_gb300.synth import make_inputs_fp8
        x8 = make_inputs_fp8(AttnShape(a.B, a.H, a.N, a.d), seed=4)
        q8, k8, v8 = (x8[n][0].cuda() for n in ("q", "k", "v"))
        sq, sk, sv = x8["q"][1], x8["k"][1], x8["v"][1]
    if a.op.endswith("blocksparse"):
        nb = (a.N + 127) // 128
        g = torch.Generator().manual_seed(3)
        mask = (torch.rand((a.H, nb, nb), generator=g) < 0.25).to(torch.uint8)
        mask[:, torch.arange(nb), torch.arange(nb)] = 1
        mask = mask.cuda()
        o, lse = attn.attn_fwd_blocksparse(q, k, v, mask, scale=scale, causal=a.causal)

    def run():
        if a.op == "fwd_fp8":
            attn.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, causal=a.causal, o=o, lse=lse)
        elif a.op == "fwd_blocksparse":
            attn.attn_fwd_blocksparse(q, k, v, mask, scale=scale, causal=a.causal, o=o, lse=lse)
        elif a.op == "bwd_blocksparse":
            attn.attn_bwd_blocksparse(q, k, v, o, do, lse, mask, scale=scale, causal=a.causal)
        elif a.op == "fwd_dropout":
            attn.attn_fwd_dropout(q, k, v, 0.1, 1234, 0, scale=scale, causal=a.causal, o=o, lse=lse)
        elif a.op == "bwd_dropout":
            attn.attn_bwd_dropout(q, k, v, o, do, lse, 0.1, 1234, 0, scale=scale, causal=a.causal)
        elif a.op == "decode":
            attn.attn_decode(q1, k, v, scale=scale)
        elif a.op == "fwd":
            attn.attn_fwd(q, k, v, scale=scale, causal=a.causal, o=o, lse=lse)
        elif a.op == "bwd":
            attn.attn_bwd(q, k, v, o, do, lse, scale=scale, causal=a.causal)
        else:
            s = torch.matmul(q, k.transpose(-2, -1)) * scale
            if a.causal:
                s = s.masked_fill(torch.ones(a.N, a.N, dtype=torch.bool, device=q.device).triu(1),
                                  float("-inf"))
            torch.matmul(torch.softmax(s, dim=-1), v)

    for _ in range(a.warmup):
        run()
    torch.cuda.synchronize()
    for _ in range(a.launches):
        run()
    torch.cuda.synchronize()
    st = attn.sync_status()
    print("done op=%s status=%d" % (a.op, st))
    return 1 if st else 0


if __name__ == "__main__":
    raise SystemExit(main())

#!/usr/bin/env python3
"""Throughput of the fused exact-attention hot path on GB300.

One step = one pass of the whole path: forward (O, LSE) then the
recomputation backward (dQ, dK, dV) on the long-sequence workload
B=2, H=16, N=8192, d=128, bf16, non-causal, scale 1/sqrt(128), with Gaussian
inputs resident in HBM.  Credited FLOPs per step are the algorithm's
matmuls only: forward 4*B*H*N^2*d, backward 2.5x that (halved for causal).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs its own copy of the workload (weak scaling:
attention heads are independent problems, so no data-path collective); the
timed region is bracketed by barriers and the max over ranks is taken.
Prints exactly one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd / fwd+bwd TFLOP/s (bf16, N=8192, d=128) and % of GB300 tensor peak"
UNIT = "TFLOP/s"
WORKLOAD = {"workload": "exact attention fwd+bwd, B=2 H=16 N=8192 d=128 bf16 non-causal, "
                        "scale 1/sqrt(128), Q/K/V/dO ~ N(0,1)",
            "B": 2, "H": 16, "N": 8192, "d": 128, "causal": False, "dtype": "bf16",
            "l2": "inputs larger than L2 (4 x 67 MB read per step; no explicit flush)"}
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def flops_per_step(B, H, N, d, causal):
    fwd = 4.0 * B * H * N * N * d
    if causal:
        fwd /= 2.0
    return fwd, 2.5 * fwd


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def shard_heads(rank, world, B, H):
    """Weak scaling: every rank owns a full, independent batch of B x H heads.
    Returns the seed offset and the global index range of this rank's heads."""
    per = B * H
    return rank, (rank * per, (rank + 1) * per)


def max_over_ranks(value, world):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {"attn_fwd_kernel": ("attn_fwd.cu", "block_order.h", "tc_sm103.cuh", "dropout.cuh"),
                  "attn_bwd_kernel": ("attn_bwd.cu", "block_order.h", "tc_sm103.cuh", "dropout.cuh"),
                  "attn_decode_split_kernel": ("attn_decode.cu", "tc_sm103.cuh")}


def code_only(text):
    """Source text without comments and with whitespace collapsed, so that an
    edit of comments alone does not count as a change of the kernel."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def sources_sha(kernel):
    """Short hash of the code (comments stripped) of the device source files a
    kernel is built from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "io_aware_exact_12_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel, config_key):
    """DRAM bytes per launch from the committed ncu summary, only if it was
    taken from the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    sha = sources_sha(kernel)
    for ln in lines:
        if ln.startswith("#") or not ln.strip():
            continue
        kv = dict(tok.split("=", 1) for tok in ln.split() if "=" in tok)
        if kv.get("kernel") == kernel and kv.get("config") == config_key and kv.get("sources_sha") == sha:
            return float(kv["dram_bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 20 ms while running.
    mark_start() / mark_end() bracket the timed region; the summary uses the
    samples taken inside it (or, for a region shorter than the sampling
    period, the samples nearest to it, and says so)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t_start = None
        self.t_end = None

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()
        time.sleep(0.05)  # let the sample that covers the end be written

    @staticmethod
    def _epoch(ts):
        import datetime
        try:
            return datetime.datetime.strptime(ts.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for ln in open(self.path).read().splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((self._epoch(parts[0]), float(parts[1]), float(parts[2]),
                             [n for n, val in zip(names, parts[5:9]) if val.lower().startswith("active")]))
            except ValueError:
                continue
        os.unlink(self.path)
        where = "all samples"
        sel = rows
        if self.t_start is not None and self.t_end is not None and all(r[0] is not None for r in rows):
            inside = [r for r in rows if self.t_start <= r[0] <= self.t_end]
            if inside:
                sel, where = inside, "inside the timed region"
            elif rows:
                mid = 0.5 * (self.t_start + self.t_end)
                sel = sorted(rows, key=lambda r: abs(r[0] - mid))[:2]
                where = "nearest to the timed region (%.0f ms, shorter than the 20 ms period)" % (
                    1e3 * (self.t_end - self.t_start))
        sm = [r[1] for r in sel]
        reasons = sorted({n for r in sel for n in r[3]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": sel[-1][2] if sel else None,
                "samples": len(sm), "which": where, "reasons": reasons}


def oracle_sample(N, d, causal, seed, heads=1):
    """Times the float64 CPU oracle (forward + analytic backward, as it
    stands) on `heads` heads of the workload.  Returns (seconds, credited
    flops, threads)."""
    import oracle
    from io_aware_exact_12_gb300.synth import AttnShape, make_inputs
    x = make_inputs(AttnShape(1, heads, N, d), "bf16", seed=seed)
    q, k, v, do = (x[n].double().numpy() for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(d)
    threads = oracle.default_threads()
    oracle.build()
    t0 = time.perf_counter()
    o, _ = oracle.forward(q, k, v, scale, causal, threads=threads)
    oracle.backward(q, k, v, o, do, scale, causal, threads=threads)
    dt = time.perf_counter() - t0
    f, b = flops_per_step(1, heads, N, d, causal)
    return dt, f + b, threads


E2E_CHUNKS = 8  # head-chunks of the pipelined end-to-end step (4 heads each at B=2 H=16)
E2E_COMPUTE_STREAMS = 8

DECODE = {"workload": "decode: 1 query token per (b, h) against a bf16 KV cache, B=16 H=16 L=32768 d=128",
          "B": 16, "H": 16, "L": 32768, "d": 128}


def measure_decode(attn, steps, warmup, peaks):
    """Decode is bound by reading the cache: report GB/s of algorithmic bytes
    (K and V once, q, o, lse) against the measured HBM copy bandwidth."""
    import torch
    B, H, L, d = DECODE["B"], DECODE["H"], DECODE["L"], DECODE["d"]
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    k = torch.randn((B, H, L, d), generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn((B, H, L, d), generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    q = torch.randn((B, H, d), generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty((B, H), device="cuda", dtype=torch.float32)
    for _ in range(max(warmup, 3)):
        attn.attn_decode(q, k, v, o=o, lse=lse)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        attn.attn_decode(q, k, v, o=o, lse=lse)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    nbytes = 2 * B * H * L * d * 2 + 2 * B * H * d * 2 + 4 * B * H
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    del k, v
    # ncu traffic was taken at L = 8192 (1.07 GB, the capture size limit); K/V traffic
    # grows in proportion to L, so it is scaled to this call's L.
    t8k = traffic_from_profiles("attn_decode_split_kernel", "b16h16l8192")
    traffic = None if t8k is None else t8k * L / 8192.0
    return dict(DECODE, ms=ms, bytes_per_call=nbytes, gbs=gbs, bound="hbm", peak_gbs=peak, frac=gbs / peak,
                traffic=traffic, traffic_note="ncu DRAM bytes at L=8192 scaled by L/8192",
                status=attn.sync_status())


def measure_exp_bound(attn, B, H, N, fwd_ms, bwd_ms):
    """Secondary bound of the softmax step: one exp2 per score, B*H*N^2 in the
    forward and as many again in the backward (recomputing P).  The rate of
    the exponential unit is measured with the library's probe kernel (the
    same ex2.approx.f32 instruction), enough blocks for 8 per SM."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    blocks, iters = sms * 8, 4096
    sink = torch.empty(blocks * attn.EX2_PROBE_THREADS, device="cuda", dtype=torch.float32)
    for _ in range(2):
        n_exp = attn.probe_ex2(sink, blocks, iters)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 5
    e0.record()
    for _ in range(reps):
        attn.probe_ex2(sink, blocks, iters)
    e1.record()
    torch.cuda.synchronize()
    rate = n_exp * reps / (e0.elapsed_time(e1) * 1e-3)  # exponentials per second
    sink_ok = bool(torch.isfinite(sink).all().item())
    exps = float(B * H * N * N)
    fwd_rate, bwd_rate = exps / (fwd_ms * 1e-3), exps / (bwd_ms * 1e-3)
    return {"unit": "exp2/s", "probe_rate": rate,
            "exps_per_pass": exps,
            "fwd": {"rate": fwd_rate, "frac": fwd_rate / rate, "floor_ms": exps / rate * 1e3},
            "bwd": {"rate": bwd_rate, "frac": bwd_rate / rate, "floor_ms": exps / rate * 1e3},
            "probe": "%d blocks x 256 threads x %d rounds x 8 chains of ex2.approx.f32" % (blocks, iters),
            "probe_output_finite": sink_ok, "status": attn.sync_status()}


def measure_fp8(attn, steps, warmup, peaks):
    """FP8 forward on the bench shape (B=2 H=16 N=8192 d=128), non-causal and
    causal, against the fp8 dense peak = measured bf16 peak x 2 (the nominal
    fp8/bf16 tensor-rate ratio, 4.5 / 2.25 PFLOP/s)."""
    import torch
    from io_aware_exact_12_gb300.synth import AttnShape, make_inputs_fp8
    B, H, N, d = WORKLOAD["B"], WORKLOAD["H"], WORKLOAD["N"], WORKLOAD["d"]
    x = make_inputs_fp8(AttnShape(B, H, N, d), seed=4)
    q8, k8, v8 = (x[n][0].cuda() for n in ("q", "k", "v"))
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    peak = 2.0 * float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    res = {"workload": "fp8 (e4m3) forward, B=2 H=16 N=8192 d=128, per-tensor descales", "peak_tflops": peak,
           "peak_source": "measured bf16 x 2 (nominal fp8/bf16 ratio)"}
    for causal in (False, True):
        def run():
            attn.attn_fwd_fp8(q8, k8, v8, x["q"][1], x["k"][1], x["v"][1], causal=causal, o=o, lse=lse)
        for _ in range(max(warmup, 3)):
            run()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            run()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        f, _ = flops_per_step(B, H, N, d, causal)
        tf = f / (ms * 1e-3) / 1e12
        res["causal" if causal else "noncausal"] = {"ms": ms, "tflops": tf, "frac": tf / peak}
    res["status"] = attn.sync_status()
    return res


def measure_blocksparse(attn, steps, warmup, peaks, density=0.25):
    """Block-sparse forward and backward on the bench shape with a seeded
    random block mask of the given density (diagonal always on).  Credited
    FLOPs count only the enabled 128 x 128 tile pairs (4 * 128 * 128 * d each
    forward, 2.5x that backward)."""
    import torch
    from io_aware_exact_12_gb300.synth import AttnShape, make_inputs
    B, H, N, d = WORKLOAD["B"], WORKLOAD["H"], WORKLOAD["N"], WORKLOAD["d"]
    nb = N // 128
    g = torch.Generator().manual_seed(3)
    mask = (torch.rand((H, nb, nb), generator=g) < density).to(torch.uint8)
    mask[:, torch.arange(nb), torch.arange(nb)] = 1
    x = make_inputs(AttnShape(B, H, N, d), "bf16", seed=4)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    m = mask.cuda()
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    g = [torch.empty_like(q) for _ in range(3)]

    def fwd():
        attn.attn_fwd_blocksparse(q, k, v, m, o=o, lse=lse)

    def bwd():
        attn.attn_bwd_blocksparse(q, k, v, o, do, lse, m, dq=g[0], dk=g[1], dv=g[2])

    pairs = int(mask.sum()) * B
    fl = 4.0 * 128 * 128 * d * pairs
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    res = {"workload": "block-sparse forward and backward, B=2 H=16 N=8192 d=128 bf16, per-head random mask",
           "density": pairs / (B * H * nb * nb)}
    for name, fn, f in (("fwd", fwd, fl), ("bwd", bwd, 2.5 * fl)):
        for _ in range(max(warmup, 3)):
            fwd()
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        res[name] = {"ms": ms, "tflops": f / (ms * 1e-3) / 1e12, "frac": f / (ms * 1e-3) / 1e12 / peak}
    res["bwd"]["traffic"] = traffic_from_profiles("attn_bwd_kernel", "c4_noncausal_blocksparse25")
    # the forward's figures also at the top level, as before
    res.update(ms=res["fwd"]["ms"], tflops=res["fwd"]["tflops"], frac=res["fwd"]["frac"])
    res["status"] = attn.sync_status()
    return res


def measure_dropout(attn, steps, warmup, peaks, p_drop=0.1):
    """Dropout forward and backward (p = 0.1, Philox draws in both kernels) on
    the bench shape, non-causal.  Credited FLOPs are those of the plain path
    (the draws add no tensor-core work): 4 B H N^2 d forward, 2.5x backward."""
    import torch
    from io_aware_exact_12_gb300.synth import AttnShape, make_inputs
    B, H, N, d = WORKLOAD["B"], WORKLOAD["H"], WORKLOAD["N"], WORKLOAD["d"]
    x = make_inputs(AttnShape(B, H, N, d), "bf16", seed=4)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    g = [torch.empty_like(q) for _ in range(3)]
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    f_fwd, f_bwd = flops_per_step(B, H, N, d, False)

    def fwd():
        attn.attn_fwd_dropout(q, k, v, p_drop, 1234, 0, o=o, lse=lse)

    def bwd():
        attn.attn_bwd_dropout(q, k, v, o, do, lse, p_drop, 1234, 0, dq=g[0], dk=g[1], dv=g[2])

    res = {"workload": "dropout p=%g, B=2 H=16 N=8192 d=128 bf16, non-causal" % p_drop}
    for name, fn, fl in (("fwd", fwd, f_fwd), ("bwd", bwd, f_bwd)):
        for _ in range(max(warmup, 3)):
            fwd()
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        tf = fl / (ms * 1e-3) / 1e12
        kern = "attn_fwd_kernel" if name == "fwd" else "attn_bwd_kernel"
        res[name] = {"ms": ms, "tflops": tf, "frac": tf / peak,
                     "traffic": traffic_from_profiles(kern, "c4_noncausal_dropout")}
    res["status"] = attn.sync_status()
    return res


def measure_small_d(attn, steps, warmup, peaks):
    """The head-dimension-64 shapes: the GPT-2 shape (B=8 H=12 N=1024 d=64,
    causal) and B=2 H=16 N=8192 d=64 (non-causal), forward and whole backward
    call (preprocess + main + dQ conversion), FLOPs as for the main workload.
    Inputs fit in L2 at the GPT-2 shape (38 MB); the number is a warm-L2 one."""
    import torch
    from io_aware_exact_12_gb300.synth import AttnShape, make_inputs
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    res = {}
    for key, (B, H, N, d, causal) in (("gpt2_shape_causal", (8, 12, 1024, 64, True)),
                                      ("n8192_d64", (2, 16, 8192, 64, False))):
        x = make_inputs(AttnShape(B, H, N, d), "bf16", seed=4)
        q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        g = [torch.empty_like(q) for _ in range(3)]
        f_fwd, f_bwd = flops_per_step(B, H, N, d, causal)

        def fwd():
            attn.attn_fwd(q, k, v, causal=causal, o=o, lse=lse)

        def bwd():
            attn.attn_bwd(q, k, v, o, do, lse, causal=causal, dq=g[0], dk=g[1], dv=g[2])

        r = {"workload": "B=%d H=%d N=%d d=%d bf16, %s" % (B, H, N, d, "causal" if causal else "non-causal")}
        for name, fn, fl in (("fwd", fwd, f_fwd), ("bwd", bwd, f_bwd)):
            for _ in range(max(warmup, 3)):
                fwd()
                fn()
            torch.cuda.synchronize()
            n = max(steps, 20)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(n):
                fn()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / n
            tf = fl / (ms * 1e-3) / 1e12
            r[name] = {"ms": ms, "tflops": tf, "frac": tf / peak}
        res[key] = r
    res["status"] = attn.sync_status()
    return res


def bench_config(world):
    """The `config` of both arms' lines (the same dict, so the two compare)."""
    return dict(WORKLOAD, parallelism="dp%d (independent heads per rank)" % world)


# Arm Ltd. (implementer 0x41) CPU part numbers of the cores these hosts carry;
# /proc/cpuinfo on Arm gives only the number.
ARM_PARTS = {0xd0c: "Neoverse-N1", 0xd40: "Neoverse-V1", 0xd49: "Neoverse-N2", 0xd4f: "Neoverse-V2",
             0xd8e: "Neoverse-N3", 0xd84: "Neoverse-V3"}


def cpu_model():
    """A readable CPU model: lscpu's model name, else /proc/cpuinfo's, else the
    Arm part number translated, with the part number beside it."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                name = ln.split(":", 1)[1].strip()
                if name and name != "-":
                    return name
    except (OSError, subprocess.SubprocessError):
        pass
    part = None
    try:
        for ln in open("/proc/cpuinfo"):
            key = ln.split(":", 1)[0].strip().lower()
            if key == "model name":
                return ln.split(":", 1)[1].strip()
            if key == "cpu part" and part is None:
                part = ln.split(":", 1)[1].strip()
    except OSError:
        pass
    if part is not None:
        try:
            return "%s (CPU part %s)" % (ARM_PARTS[int(part, 16)], part)
        except (KeyError, ValueError):
            return "CPU part %s" % part
    import platform
    return platform.machine()


def run_reference(args):
    """The oracle arm: the float64 CPU oracle timed on the host cores, each
    step one head (of 32) of the same workload, forward + backward."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    N, d, causal = WORKLOAD["N"], WORKLOAD["d"], WORKLOAD["causal"]
    times, fl, threads = [], 0.0, 1
    for i in range(args.warmup + args.steps):
        dt, fl, threads = oracle_sample(N, d, causal, seed=100 + i, heads=1)
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = fl * len(times) / total / 1e12
    sample = "1 of 32 heads (B=1, H=1, N=8192, d=128, non-causal) per step, forward + backward"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": bench_config(world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample, "cpu": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from io_aware_exact_12_gb300 import build as build_mod
    if rank == 0 or not os.path.exists(build_mod.LIB_PATH):
        build_mod.build()
    barrier(world)
    import io_aware_exact_12_gb300 as attn
    from io_aware_exact_12_gb300.synth import AttnShape, make_inputs

    B, H, N, d, causal = (WORKLOAD[k] for k in ("B", "H", "N", "d", "causal"))
    scale = 1.0 / math.sqrt(d)
    seed_off, _ = shard_heads(rank, world, B, H)
    host = make_inputs(AttnShape(B, H, N, d), "bf16", seed=4 + seed_off)
    q, k, v, do = (host[n].cuda() for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    stream = torch.cuda.current_stream()

    def step(c=causal):
        attn.attn_fwd(q, k, v, scale=scale, causal=c, o=o, lse=lse)
        attn.attn_bwd(q, k, v, o, do, lse, scale=scale, causal=c, dq=dq, dk=dk, dv=dv)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if attn.sync_status() != 0:
        raise SystemExit("device status error during warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        clocks.mark_start()
        for i in range(K):
            ev[i][0].record(stream)
            attn.attn_fwd(q, k, v, scale=scale, causal=causal, o=o, lse=lse)
            ev[i][1].record(stream)
            attn.attn_bwd(q, k, v, o, do, lse, scale=scale, causal=causal, dq=dq, dk=dk, dv=dv)
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        clocks.mark_end()
        barrier(world)
    status = attn.sync_status()
    clk = clocks.summary()
    total_ms = ev[0][0].elapsed_time(ev[K - 1][2])
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    ms_step = max_over_ranks(total_ms / K, world)
    f_fwd, f_bwd = flops_per_step(B, H, N, d, causal)
    value = world * (f_fwd + f_bwd) / (ms_step * 1e-3) / 1e12
    launches = K * 4
    dv_ref_last = dv.view(B * H, N, d)[-1].clone()  # the timed steps' dV of the last head (checks e2e below)

    # causal variant of the same workload (reported alongside, not in `value`),
    # timed like the main step: back-to-back steps, one synchronisation at the end
    for _ in range(3):
        step(True)
    torch.cuda.synchronize()
    cev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(max(K // 2, 3))]
    for e0, e1, e2 in cev:
        e0.record(stream)
        attn.attn_fwd(q, k, v, scale=scale, causal=True, o=o, lse=lse)
        e1.record(stream)
        attn.attn_bwd(q, k, v, o, do, lse, scale=scale, causal=True, dq=dq, dk=dk, dv=dv)
        e2.record(stream)
    torch.cuda.synchronize()
    cf_ms = [e0.elapsed_time(e1) for e0, e1, _ in cev]
    cb_ms = [e1.elapsed_time(e2) for _, e1, e2 in cev]
    cf_f, cb_f = flops_per_step(B, H, N, d, True)

    # end to end through the public API: pinned host inputs -> device -> fwd+bwd -> host outputs
    hin = {n: host[n].pin_memory() for n in ("q", "k", "v", "do")}
    hout = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    h2d = sum(t.numel() * t.element_size() for t in hin.values())
    d2h = sum(t.numel() * t.element_size() for t in hout.values())

    def e2e_step_sequential():
        q.copy_(hin["q"], non_blocking=True)
        k.copy_(hin["k"], non_blocking=True)
        v.copy_(hin["v"], non_blocking=True)
        do.copy_(hin["do"], non_blocking=True)
        step()
        hout["o"].copy_(o, non_blocking=True)
        hout["lse"].copy_(lse, non_blocking=True)
        hout["dq"].copy_(dq, non_blocking=True)
        hout["dk"].copy_(dk, non_blocking=True)
        hout["dv"].copy_(dv, non_blocking=True)

    # Pipelined: heads are independent, so the step runs over E2E_CHUNKS groups
    # of heads; chunk c+1's inputs are copied in (stream s_in) while chunk c
    # computes (E2E_COMPUTE_STREAMS compute streams in turn, so one chunk's
    # kernels can fill the SMs the previous chunk's leave idle at their tail) and
    # chunk c-1's results are copied out (stream s_out).  Every input byte is
    # copied in and every result byte copied out inside the step.  The pinned
    # host buffers hold each chunk's q, k, v, dO (and o, dq, dk, dv) next to one
    # another, so a chunk moves in one copy and out in two (o/dq/dk/dv, lse),
    # and the per-chunk tensors and events are made once, outside the timed
    # region: the host's work per step stays well below the GPU's.
    BH = B * H
    nch = args.e2e_chunks if args.e2e_chunks > 0 and BH % args.e2e_chunks == 0 else 1
    hc = BH // nch
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    s_cmp = [torch.cuda.Stream() for _ in range(max(1, args.e2e_streams))]

    def flat(t):
        return t.view(BH, *t.shape[2:])

    IN_NAMES, OUT_NAMES = ("q", "k", "v", "do"), ("o", "dq", "dk", "dv")
    hin_pk = torch.empty((nch, 4, hc, N, d), dtype=q.dtype, pin_memory=True)
    for j, n in enumerate(IN_NAMES):
        hin_pk[:, j].copy_(flat(hin[n]).view(nch, hc, N, d))
    # Two sets of device buffers (and of pinned host outputs): step i uses set
    # i % 2, so step i+1's input copies overlap step i's compute and copies out,
    # and step i+2 waits for step i to have finished with the set.
    sets = []
    for sidx in range(2):
        din = torch.empty((nch, 4, hc, N, d), dtype=q.dtype, device=q.device)
        dout = torch.empty((nch, 4, hc, N, d), dtype=q.dtype, device=q.device)
        dlse = torch.empty((nch, hc, N), dtype=lse.dtype, device=q.device)
        hout_pk = torch.empty((nch, 4, hc, N, d), dtype=q.dtype, pin_memory=True)
        hlse = torch.empty((nch, hc, N), dtype=lse.dtype, pin_memory=True)
        views = [{**{n: din[c, j].unsqueeze(0) for j, n in enumerate(IN_NAMES)},
                  **{n: dout[c, j].unsqueeze(0) for j, n in enumerate(OUT_NAMES)},
                  "lse": dlse[c].unsqueeze(0)} for c in range(nch)]
        sets.append({"din": din, "dout": dout, "dlse": dlse, "hout": hout_pk, "hlse": hlse, "views": views,
                     "ev_in": [torch.cuda.Event() for _ in range(nch)],
                     "ev_cmp": [torch.cuda.Event() for _ in range(nch)], "done": torch.cuda.Event()})

    def e2e_step(start_ev, sidx=0):
        st = sets[sidx]
        s_in.wait_event(start_ev)
        with torch.cuda.stream(s_in):
            for c in range(nch):
                st["din"][c].copy_(hin_pk[c], non_blocking=True)
                st["ev_in"][c].record(s_in)
        for c in range(nch):
            sc = s_cmp[c % len(s_cmp)]
            sc.wait_event(st["ev_in"][c])
            w = st["views"][c]
            with torch.cuda.stream(sc):
                attn.attn_fwd(w["q"], w["k"], w["v"], scale=scale, causal=causal, o=w["o"], lse=w["lse"])
                attn.attn_bwd(w["q"], w["k"], w["v"], w["o"], w["do"], w["lse"], scale=scale, causal=causal,
                              dq=w["dq"], dk=w["dk"], dv=w["dv"])
                st["ev_cmp"][c].record(sc)
        with torch.cuda.stream(s_out):
            for c in range(nch):
                s_out.wait_event(st["ev_cmp"][c])
                st["hout"][c].copy_(st["dout"][c], non_blocking=True)
                st["hlse"][c].copy_(st["dlse"][c], non_blocking=True)
        st["done"].record(s_out)
        stream.wait_event(st["done"])
        return st["done"]

    def time_e2e(fn, sets):
        # With one buffer set each step starts after the previous one has
        # finished (its input copies overwrite the buffers the previous step
        # computed from); with two, after the step two back has finished.
        for _ in range(max(args.warmup, 3)):
            w = torch.cuda.Event()
            w.record(stream)
            fn(w, 0)
        torch.cuda.synchronize()
        barrier(world)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        done = [s0] * sets
        for i in range(K):
            done[i % sets] = fn(done[i % sets], i % sets) or done[i % sets]
        for e in done:
            stream.wait_event(e)
        s1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(s0.elapsed_time(s1) / K, world)

    e2e_ms = time_e2e(e2e_step, 2)
    e2e_value = world * (f_fwd + f_bwd) / (e2e_ms * 1e-3) / 1e12
    launches_e2e = K * 4 * nch
    # Checks on the last head's dV (no atomics in dV): each host copy equals the
    # device buffer it was copied from, both buffer sets hold the same numbers,
    # and they equal the timed steps' dV to rounding (a chunk of 4 heads makes
    # a grid without the full grid's split last wave, so the fp32 partial sums
    # of the split key tiles associate differently).
    last = [st["hout"][nch - 1, 3, hc - 1] for st in sets[:min(2, K)]]
    e2e_check = (all(bool(torch.equal(h.cuda(), st["dout"][nch - 1, 3, hc - 1])) for h, st in zip(last, sets))
                 and all(bool(torch.equal(h, last[0])) for h in last)
                 and bool(torch.allclose(last[0].cuda().float(), dv_ref_last.float(), rtol=1e-2, atol=1e-3)))
    seq_ms = time_e2e(lambda ev, sidx: e2e_step_sequential(), 1)  # one stream: already serialised

    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    fwd_tf = f_fwd / (fwd_ms * 1e-3) / 1e12
    bwd_tf = f_bwd / (bwd_ms * 1e-3) / 1e12
    # dominant kernel: the one with the larger share of the step
    if bwd_ms >= fwd_ms:
        dom, dom_tf, dom_name = "attn_bwd_kernel", bwd_tf, "bwd"
    else:
        dom, dom_tf, dom_name = "attn_fwd_kernel", fwd_tf, "fwd"
    traffic = traffic_from_profiles(dom, "c4_noncausal")
    roof = {"bound": "tensor", "kernel": dom, "achieved": dom_tf, "peak": peak, "unit": UNIT,
            "frac": dom_tf / peak, "traffic": traffic, "peak_source": peak_src + " (burst bf16)",
            "frac_of_sustained": dom_tf / peak_sus,
            "note": ("bwd duration is the whole attn_bwd call (preprocess + main + dQ convert), "
                     "so `achieved` understates the main kernel slightly") if dom_name == "bwd" else ""}

    decode = measure_decode(attn, K, args.warmup, peaks) if rank == 0 else None
    fp8 = measure_fp8(attn, K, args.warmup, peaks) if rank == 0 else None
    sparse = measure_blocksparse(attn, K, args.warmup, peaks) if rank == 0 else None
    dropout = measure_dropout(attn, K, args.warmup, peaks) if rank == 0 else None
    small_d = measure_small_d(attn, K, args.warmup, peaks) if rank == 0 else None
    exp_bound = measure_exp_bound(attn, B, H, N, fwd_ms, bwd_ms) if rank == 0 else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, fl, threads = oracle_sample(N, d, causal, seed=4, heads=5)
        cpu = {"value": fl / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": "5 of 32 heads (B=1, H=5, N=8192, d=128, non-causal), forward + backward, "
                         "%.1f s" % dt, "cpu": cpu_model()}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": bench_config(world),
                "fwd": {"ms": fwd_ms, "tflops": fwd_tf, "frac_of_peak": fwd_tf / peak},
                "bwd": {"ms": bwd_ms, "tflops": bwd_tf, "frac_of_peak": bwd_tf / peak},
                "causal": {"fwd_ms": statistics.median(cf_ms), "bwd_ms": statistics.median(cb_ms),
                           "fwd_tflops": cf_f / (statistics.median(cf_ms) * 1e-3) / 1e12,
                           "bwd_tflops": cb_f / (statistics.median(cb_ms) * 1e-3) / 1e12},
                "roofline": roof, "cpu_baseline": cpu, "decode": decode, "fp8": fp8, "blocksparse": sparse,
                "dropout": dropout, "d64": small_d, "exp_bound": exp_bound,
                "e2e": {"value": e2e_value, "unit": UNIT, "ms_per_step": e2e_ms,
                        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                        "pipeline": ("%d head-chunks: copies in / compute (%d streams) / copies out overlapped; "
                                     "consecutive steps overlap on two device buffer sets" % (
                                         nch, len(s_cmp))),
                        "sequential_ms_per_step": seq_ms,
                        "sequential_value": world * (f_fwd + f_bwd) / (seq_ms * 1e-3) / 1e12,
                        "outputs_match_device": e2e_check},
                "gpu_launches": launches, "gpu_launches_e2e": launches_e2e,
                "clocks": clk, "device_status": status}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=E2E_CHUNKS,
                    help="head-chunks of the pipelined end-to-end step (must divide B*H, else 1)")
    ap.add_argument("--e2e-streams", type=int, default=E2E_COMPUTE_STREAMS,
                    help="compute streams the end-to-end chunks rotate over")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

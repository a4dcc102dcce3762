"""Benchmark of the emulated-FP32 GEMM on GB300: prints one JSON line.

Metric: effective FP32 TFLOP/s = 2MNK / t, also as a fraction of the dense
BF16 tensor peak / 9 (nine BF16 products per emulated FP32 product).  A step
is one emu_sgemm call -- the whole hot path: split of A, split of B, the
tensor-core GEMM with its epilogue -- on inputs already resident in HBM.

Default workload: C = A B with A, B 8192 x 8192 drawn from N(0, 1), BF16x9,
beta = 0 (the size at which the method's square-GEMM speedups are quoted).
Each operand is 256 MiB, larger than the 129 MB L2, so no flush is needed
between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--mode bf16x9|tf32x3|tf32x3_oy|bf16x3|tf32|fp32_simt] [--impl reference]

--impl reference times the CPU oracle (the plain reference implementation of
the method) on the host cores, on a bounded block of rows of the same
workload, and prints the same metric.  Under torchrun (N > 1) every rank runs
an independent replica on its own GPU (the GEMM does not exchange data);
value is the total over ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "emulated-FP32 GEMM TFLOP/s (2MNK/t) and % of BF16 dense peak/9 on 1 GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float) -> float:
    """The maximum of x over all ranks (x itself when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: float, world: int, steps: int, ms_total: float) -> float:
    """Whole-job TFLOP/s: every rank runs `steps` steps of `flops_per_step`;
    the job takes as long as its slowest rank (ms_total is that maximum)."""
    return flops_per_step * world * steps / (ms_total * 1e-3) / 1e12


# ------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r[2] > 200.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows),
                "samples": len(loaded),
                "reasons": reasons}


# ------------------------------------------------------------- GPU arm --

def bench_gpu(args):
    import numpy as np
    import torch

    from fp32_emulated_gemm_split_gb300 import _build
    from fp32_emulated_gemm_split_gb300 import workloads as W

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    _build.build()
    import fp32_emulated_gemm_split_gb300 as emu
    if args.path:
        emu.emu_set_path(args.path)

    g = pick_workload(W, args)
    A, B, C0 = W.generate(g)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C0).cuda() if C0 is not None else torch.empty((g.M, g.N), device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        emu.emu_sgemm(dA, dB, dC, transA=g.transA, transB=g.transB, alpha=g.alpha, beta=g.beta,
                      mode=g.mode, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    emu.emu_profile_enable(True)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        start.record(stream)
        for _ in range(args.steps):
            step()
        stop.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
    ms_total = start.elapsed_time(stop)
    prof = {k: emu.emu_profile_read(k) for k in ("split", "gemm_tc", "gemm_fused", "gemm_simt", "scale")}
    emu.emu_profile_enable(False)
    assert emu.emu_get_last_device_error() == 0, "device-side wait gave up during the bench"

    ms_total = max_over_ranks(ms_total)
    ms_step = ms_total / args.steps
    flops = g.flops
    value = job_throughput(flops, world, args.steps, ms_total)
    peaks, peak_src = load_peaks()
    p_bf16 = float(peaks["bf16_tflops"])
    frac9 = value / world / (p_bf16 / 9.0)

    # dominant kernel: the tensor-core GEMM (or the SIMT kernel in that mode)
    launches = sum(n for n, _ in prof.values())
    if g.mode == "fp32_simt":
        dom_name, (n_dom, ms_dom) = "gemm_simt", prof["gemm_simt"]
    elif prof["gemm_fused"][0] > 0:
        dom_name, (n_dom, ms_dom) = "gemm_fused", prof["gemm_fused"]
    else:
        dom_name, (n_dom, ms_dom) = "gemm_tc", prof["gemm_tc"]
    per_launch_ms = ms_dom / max(n_dom, 1)
    products = {"bf16x9": 9, "tf32x3": 3, "tf32x3_oy": 3, "bf16x3": 3, "tf32": 1,
                "fp32_simt": 1}[g.mode]
    tf32_mode = g.mode in ("tf32x3", "tf32x3_oy", "tf32")
    if g.mode == "fp32_simt":
        roofline = {"bound": "alu", "achieved": flops / (per_launch_ms * 1e-3) / 1e12,
                    "peak": None, "unit": "TFLOP/s", "frac": None, "traffic": None}
    else:
        # tensor FLOPs per launch: products * 2MNK; TF32 runs at half the BF16 rate
        tensor_flops = products * flops
        achieved = tensor_flops / (per_launch_ms * 1e-3) / 1e12
        peak = p_bf16 / 2.0 if tf32_mode else p_bf16
        roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
                    "kernel": dom_name,
                    "peak_source": f"{peak_src} bf16 burst" + (" / 2 (tf32 nominal ratio)" if tf32_mode else ""),
                    "kernel_ms": round(per_launch_ms, 4)}
        traffic = load_traffic(dom_name, g.name, g.mode)
        if traffic is not None:
            roofline["traffic"] = traffic

    split_n, split_ms = prof["split"]
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": g.name, "M": g.M, "N": g.N, "K": g.K, "mode": g.mode,
                   "transA": g.transA, "transB": g.transB, "alpha": g.alpha, "beta": g.beta,
                   "path": emu.emu_get_path(), "emulates": "fp32",
                   "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas{world}"},
        "pct_of_bf16_peak_over_9": round(100.0 * frac9, 2),
        "bf16_peak_tflops": p_bf16,
        "roofline": roofline,
        "kernels": {"split_ms_per_step": round(split_ms / args.steps, 4),
                    f"{dom_name}_ms_per_launch": round(per_launch_ms, 4)},
        "gpu_launches": launches,
    }
    out["clocks"] = clocks.summary()

    if rank == 0:
        if not args.no_configs:
            del dA, dB, dC
            torch.cuda.empty_cache()
            out["configs"] = bench_configs(emu, stream, peaks, peak_src)
            out["ladder"] = bench_ladder(emu, stream, peaks, peak_src)
            out["weight_gradients"] = bench_weight_gradients(emu, stream, peaks, peak_src)
            dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
            dC = torch.from_numpy(C0).cuda() if C0 is not None else torch.empty((g.M, g.N), device="cuda")
        if not args.no_e2e:
            out["e2e"] = bench_e2e(emu, g, A, B, C0, stream, args)
        if not args.no_simt and g.mode != "fp32_simt":
            out["simt_fp32"] = bench_simt(emu, g, dA, dB, dC, stream)
        if not args.no_cpu:
            out["cpu_baseline"] = cpu_baseline(g, A, B, C0, args.cpu_seconds)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


# ------------------------------------------------------ every config --

# The benchmark's configurations besides the headline one: the 256^3 GEMM,
# the three linear layers of a transformer interatomic potential on the
# edge tokens of a 192-atom and of a 17,280-atom system (M = atoms x 64),
# the dynamic-range stress GEMM with alpha and beta, and the 8192^3 GEMM in
# TF32x3 mode.
CONFIG_WORKLOADS = ["square256_uniform",
                    "mlip192_k256_n256", "mlip192_k256_n1024", "mlip192_k1024_n256",
                    "mlip17280_k256_n256", "mlip17280_k256_n1024", "mlip17280_k1024_n256",
                    "stress4096", "square8192_normal_tf32x3"]


def device_operands(g):
    """A, B (and C0) of workload g drawn on the GPU with a seeded torch
    generator: the distributions of the workload (workloads.py), not its
    exact values (drawing 4.5 GB on the host would take minutes)."""
    import torch
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1000 + g.seed)
    a_shape = (g.K, g.M) if g.transA else (g.M, g.K)
    b_shape = (g.N, g.K) if g.transB else (g.K, g.N)

    def normal(shape, std=1.0):
        x = torch.randn(shape, generator=gen, device="cuda")
        return x.mul_(std) if std != 1.0 else x

    def uniform(shape):
        return torch.rand(shape, generator=gen, device="cuda").mul_(2.0).sub_(1.0)

    def stress(shape):
        # sign * m * 2^e, m ~ U[1, 2), e ~ U{-30..30}; 1% zeros, 0.1% subnormals
        n = 1
        for d in shape:
            n *= d
        sign = torch.where(torch.rand(n, generator=gen, device="cuda") < 0.5, -1.0, 1.0)
        m = torch.rand(n, generator=gen, device="cuda").add_(1.0)
        e = torch.randint(-30, 31, (n,), generator=gen, device="cuda", dtype=torch.int32)
        x = torch.ldexp(sign * m, e.float())
        u = torch.rand(n, generator=gen, device="cuda")
        x[u < 0.01] = 0.0
        bits = torch.randint(1, 1 << 23, (n,), generator=gen, device="cuda", dtype=torch.int32)
        bits = bits | torch.where(sign < 0, torch.tensor(-(1 << 31), dtype=torch.int32, device="cuda"),
                                  torch.tensor(0, dtype=torch.int32, device="cuda"))
        sub = (u >= 0.01) & (u < 0.011)
        x[sub] = bits.view(torch.float32)[sub]
        return x.view(shape)

    if g.dist == "mlip":
        return normal(a_shape), normal(b_shape, g.K ** -0.5), None
    draw = {"normal": normal, "uniform": uniform, "stress": stress}[g.dist]
    A, B = draw(a_shape), draw(b_shape)
    C0 = uniform((g.M, g.N)) if g.beta != 0.0 else None
    return A, B, C0


def bench_configs(emu, stream, peaks, peak_src, reps=10):
    """Each configuration timed two ways: single calls on a cold L2 (a 256 MB
    buffer is written between calls, outside the timed region; the median of
    `reps` calls, CUDA events around each call on the launching stream), and
    `reps` calls back to back (the steady state of consecutive layers, events
    around the run).  Single calls are compared with the burst BF16 peak,
    back-to-back runs with the sustained one (MEASURED_PEAKS.json).  The
    dominant kernel's time per launch comes from the library's own events."""
    import torch
    from fp32_emulated_gemm_split_gb300 import workloads as W
    p_bf16 = float(peaks["bf16_tflops"])
    p_sus = float(peaks.get("bf16_tflops_sustained", p_bf16))
    # L2 flush between single calls: write a 256 MB buffer (> L2), then read
    # another, so that the flush's dirty lines are written back before the
    # timed call rather than during it
    flush = torch.empty(64 << 20, dtype=torch.float32, device="cuda")
    flush_r = torch.zeros(64 << 20, dtype=torch.float32, device="cuda")
    res = {}
    for name in CONFIG_WORKLOADS:
        g = W.WORKLOADS[name]
        A, B, C0 = device_operands(g)
        C = C0.clone() if C0 is not None else torch.empty((g.M, g.N), device="cuda")

        def call():
            emu.emu_sgemm(A, B, C, transA=g.transA, transB=g.transB, alpha=g.alpha, beta=g.beta,
                          mode=g.mode, stream=stream)

        for _ in range(3):
            call()
        torch.cuda.synchronize()
        emu.emu_profile_enable(True)
        evs = []
        for _ in range(reps):
            flush.zero_()
            flush_r.sum()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            call()
            e.record(stream)
            evs.append((s, e))
        torch.cuda.synchronize()
        prof = {k: emu.emu_profile_read(k) for k in ("split", "gemm_tc", "gemm_fused", "gemm_simt")}
        emu.emu_profile_enable(False)
        single = statistics.median(s.elapsed_time(e) for s, e in evs)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(reps):
            call()
        e.record(stream)
        torch.cuda.synchronize()
        b2b = s.elapsed_time(e) / reps
        dom = "gemm_fused" if prof["gemm_fused"][0] > 0 else "gemm_tc"
        n_dom, ms_dom = prof[dom]
        k_ms = ms_dom / max(n_dom, 1)
        products = {"bf16x9": 9, "tf32x3": 3}[g.mode]
        tf32 = g.mode == "tf32x3"
        peak = p_bf16 / 2.0 if tf32 else p_bf16
        entry = {
            "M": g.M, "N": g.N, "K": g.K, "mode": g.mode, "transB": g.transB,
            "alpha": g.alpha, "beta": g.beta,
            "path": "on-chip split of A" if dom == "gemm_fused" else "two-pass",
            "value": round(g.flops / (single * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms": round(single, 4),
            "pct_bf16_peak_over_9": round(100.0 * g.flops / (single * 1e-3) / 1e12 / (p_bf16 / 9), 1),
            "b2b_value": round(g.flops / (b2b * 1e-3) / 1e12, 2), "b2b_ms": round(b2b, 4),
            "b2b_pct_sustained_peak_over_9": round(
                100.0 * g.flops / (b2b * 1e-3) / 1e12 / (p_sus / 9), 1),
            "kernel": dom, "kernel_ms": round(k_ms, 4),
            "kernel_frac": round(products * g.flops / (k_ms * 1e-3) / 1e12 / peak, 4),
            "split_ms": round(prof["split"][1] / max(reps, 1), 4),
        }
        if tf32:
            entry["pct_bf16_peak_over_6"] = round(
                100.0 * g.flops / (single * 1e-3) / 1e12 / (p_bf16 / 6), 1)
        if g.dist == "mlip":
            # the layer's weight split once and reused (emu_sgemm_bsplit):
            # what a linear layer applied batch after batch runs
            P = emu.emu_split_b(B, transB=g.transB, mode=g.mode)

            def call_ws():
                emu.emu_sgemm_bsplit(A, P, C, transA=g.transA, alpha=g.alpha, beta=g.beta,
                                     mode=g.mode, stream=stream)

            for _ in range(3):
                call_ws()
            torch.cuda.synchronize()
            evs = []
            for _ in range(reps):
                flush.zero_()
                flush_r.sum()
                s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s.record(stream)
                call_ws()
                e.record(stream)
                evs.append((s, e))
            torch.cuda.synchronize()
            ws_single = statistics.median(s.elapsed_time(e) for s, e in evs)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            for _ in range(reps):
                call_ws()
            e.record(stream)
            torch.cuda.synchronize()
            ws_b2b = s.elapsed_time(e) / reps
            entry["weight_split_once"] = {
                "value": round(g.flops / (ws_single * 1e-3) / 1e12, 2), "ms": round(ws_single, 4),
                "pct_bf16_peak_over_9": round(
                    100.0 * g.flops / (ws_single * 1e-3) / 1e12 / (p_bf16 / 9), 1),
                "b2b_value": round(g.flops / (ws_b2b * 1e-3) / 1e12, 2), "b2b_ms": round(ws_b2b, 4),
                "b2b_pct_sustained_peak_over_9": round(
                    100.0 * g.flops / (ws_b2b * 1e-3) / 1e12 / (p_sus / 9), 1),
                "api": "emu_sgemm_bsplit"}
            del P
        res[name] = entry
        del A, B, C, C0
        torch.cuda.empty_cache()
    res["_how"] = ("operands drawn on the GPU (seeded torch generator, the workloads' "
                   "distributions); value: median of single calls with L2 flushed before each "
                   "(a 256 MB buffer written, another read) "
                   f"(% of burst P/9, {peak_src}); b2b: calls back to back (% of sustained P/9); "
                   "kernel_frac: tensor FLOPs per launch / kernel time / peak "
                   "(TF32: half the BF16 peak); weight_split_once: the layer's weight split "
                   "once (emu_split_b) and every call through emu_sgemm_bsplit")
    return res


# The accuracy ladder on one shape: every tensor-core mode of the library,
# its tensor products per emulated FP32 product and whether it runs on the
# TF32 datapath (half the BF16 rate).
LADDER = {"bf16x9": (9, False), "tf32x3": (3, True), "tf32x3_oy": (3, True),
          "bf16x3": (3, False), "tf32": (1, True)}


def bench_ladder(emu, stream, peaks, peak_src, reps=10):
    """Every tensor-core mode on the 8192^3 workload's operands (drawn on the
    GPU), 10 calls back to back: effective FP32 TFLOP/s, the dominant
    kernel's tensor throughput over its own datapath's peak (the mode's
    products per FP32 product; TF32 against half the BF16 peak), and the
    relative error on 4096 sampled outputs against an FP64 product of the
    same operands."""
    import torch
    from fp32_emulated_gemm_split_gb300 import workloads as W
    p_bf16 = float(peaks["bf16_tflops"])
    g = W.WORKLOADS["square8192_normal"]
    A, B, _ = device_operands(g)
    C = torch.empty((g.M, g.N), device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(77)
    mi = torch.randint(0, g.M, (4096,), generator=gen, device="cuda")
    ni = torch.randint(0, g.N, (4096,), generator=gen, device="cuda")
    ref = (A[mi].double() * B[:, ni].t().double()).sum(1)
    res = {}
    for mode, (products, tf32) in LADDER.items():
        run = lambda: emu.emu_sgemm(A, B, C, mode=mode, stream=stream)
        for _ in range(3):
            run()
        torch.cuda.synchronize()
        emu.emu_profile_enable(True)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(reps):
            run()
        e.record(stream)
        torch.cuda.synchronize()
        n, ms = emu.emu_profile_read("gemm_tc")
        emu.emu_profile_enable(False)
        step = s.elapsed_time(e) / reps
        k_ms = ms / max(n, 1)
        peak = p_bf16 / 2.0 if tf32 else p_bf16
        got = C[mi, ni].double()
        res[mode] = {
            "value": round(g.flops / (step * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms": round(step, 4), "kernel_ms": round(k_ms, 4),
            "kernel_frac": round(products * g.flops / (k_ms * 1e-3) / 1e12 / peak, 4),
            "rel_error": float(f"{float((got - ref).norm() / ref.norm()):.3e}"),
        }
    res["_how"] = ("square8192_normal operands drawn on the GPU; 10 calls back to back; "
                   "kernel_frac: products x 2MNK / kernel time / peak "
                   f"({peak_src} BF16 burst; TF32 modes: half of it); rel_error: relative "
                   "Frobenius error on 4096 sampled outputs against FP64")
    del A, B, C
    torch.cuda.empty_cache()
    return res


def bench_weight_gradients(emu, stream, peaks, peak_src, reps=5):
    """The weight gradients of the 17,280-atom MLIP layers, dW = dY^T X over
    their 1,105,920 rows (what EmuLinear's backward computes): M x N x K =
    256 x 256 x 1105920 and 1024 x 256 x 1105920, op(A) = dY^T (transA),
    BF16x9, operands drawn on the GPU, `reps` calls back to back.  A few
    output tiles with K blocks in the thousands: the GEMM's tail spreads
    them over every SM pair."""
    import torch
    p_bf16 = float(peaks["bf16_tflops"])
    gen = torch.Generator(device="cuda")
    gen.manual_seed(2024)
    res = {}
    for (M, N, K) in [(256, 256, 1105920), (1024, 256, 1105920)]:
        dY = torch.randn((K, M), generator=gen, device="cuda")
        X = torch.randn((K, N), generator=gen, device="cuda").mul_(K ** -0.5)
        C = torch.empty((M, N), device="cuda")
        run = lambda: emu.emu_sgemm(dY, X, C, transA=True, stream=stream)
        for _ in range(2):
            run()
        torch.cuda.synchronize()
        emu.emu_profile_enable(True)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(reps):
            run()
        e.record(stream)
        torch.cuda.synchronize()
        n, ms = emu.emu_profile_read("gemm_tc")
        ns, mss = emu.emu_profile_read("split")
        emu.emu_profile_enable(False)
        step = s.elapsed_time(e) / reps
        flops = 2.0 * M * N * K
        k_ms = ms / max(n, 1)
        res[f"{M}x{N}x{K}"] = {
            "value": round(flops / (step * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms": round(step, 4), "kernel_ms": round(k_ms, 4),
            "kernel_frac": round(9 * flops / (k_ms * 1e-3) / 1e12 / p_bf16, 4),
            "split_ms": round(mss / reps, 4),
        }
        del dY, X, C
        torch.cuda.empty_cache()
    res["_how"] = ("dW = dY^T X of the 1.1M-row MLIP layers (transA), BF16x9, operands drawn "
                   "on the GPU, 5 calls back to back; kernel_frac: 18MNK / GEMM time / "
                   f"{peak_src} BF16 burst peak; split_ms: both operands' splits (row-wise, "
                   "into M- and N-major pieces)")
    return res


def pick_workload(W, args):
    """The named workload, optionally with another mode or another M,N,K
    (same value distribution) for small profiling runs."""
    from dataclasses import replace
    base = W.WORKLOADS[args.workload]
    g = W.with_mode(base, args.mode or base.mode)
    if args.shape:
        M, N, K = (int(v) for v in args.shape.split(","))
        g = replace(g, name=f"{base.name}@{M}x{N}x{K}", M=M, N=N, K=K)
    return g


def load_traffic(kernel, workload, mode):
    """DRAM bytes per launch of `kernel` from a committed ncu capture
    (profiles/traffic.json), if one matches this kernel, workload and mode and
    none of the sources it records (the kernel, and the host code that picks
    its operands' layouts) has changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(f"{kernel}:{workload}:{mode}")
    if not rec:
        return None
    for rel, sha in rec["sources"].items():
        src = os.path.join(ROOT, rel)
        if not os.path.exists(src):
            return None
        with open(src, "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != sha:
                return None
    return rec["bytes"]


def bench_e2e(emu, g, A, B, C0, stream, args):
    """Same metric through emu_sgemm_host: host->device copies of A and B (and
    C0), the GEMM and the device->host copy of C inside the timed region."""
    import numpy as np
    import torch
    pa = torch.empty(A.shape, dtype=torch.float32, pin_memory=True).numpy()
    pb = torch.empty(B.shape, dtype=torch.float32, pin_memory=True).numpy()
    pc = torch.empty((g.M, g.N), dtype=torch.float32, pin_memory=True).numpy()
    pa[...] = A
    pb[...] = B
    if C0 is not None:
        pc[...] = C0

    def once():
        emu.emu_sgemm_host(pa, pb, pc, transA=g.transA, transB=g.transB, alpha=g.alpha,
                           beta=g.beta, mode=g.mode, stream=stream)

    once()
    steps = max(2, min(args.steps, 5))
    t0 = time.perf_counter()
    for _ in range(steps):
        once()
    dt = (time.perf_counter() - t0) / steps
    h2d = (A.size + B.size + (C0.size if C0 is not None else 0)) * 4
    return {"value": round(g.flops / dt / 1e12, 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(g.M * g.N * 4),
            "ms_per_step": round(dt * 1e3, 3), "api": "emu_sgemm_host", "memory": "pinned"}


def bench_simt(emu, g, dA, dB, dC, stream):
    """The library's own FP32 SIMT kernel on the same operands (context)."""
    import torch
    run = lambda: emu.emu_sgemm(dA, dB, dC, transA=g.transA, transB=g.transB, alpha=g.alpha,
                                beta=g.beta, mode="fp32_simt", stream=stream)
    run()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = 3
    s.record(stream)
    for _ in range(n):
        run()
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / n
    return {"value": round(g.flops / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "ms_per_call": round(ms, 3)}


def ORACLE_FN(oracle):
    return {"bf16x9": oracle.gemm_bf16x9, "tf32x3": oracle.gemm_tf32x3,
            "tf32x3_oy": oracle.gemm_tf32x3_oy,
            "bf16x3": oracle.gemm_bf16x3, "tf32": oracle.gemm_tf32,
            "fp32_simt": oracle.gemm_fp32}


def cpu_baseline(g, A, B, C0, seconds):
    """The CPU oracle (plain C, OpenMP over the host cores) on a block of rows
    of the same GEMM, scaled to the metric's unit."""
    import numpy as np
    import oracle
    fn = ORACLE_FN(oracle)[g.mode]
    threads = oracle.max_threads()

    def rows_pairs(r):
        mi = np.repeat(np.arange(r, dtype=np.int64), g.N)
        ni = np.tile(np.arange(g.N, dtype=np.int64), r)
        return mi, ni

    r = 1
    t0 = time.perf_counter()
    fn(A, B, g.transA, g.transB, g.alpha, g.beta, C0, pairs=rows_pairs(r))
    t1 = time.perf_counter() - t0
    # size the sample to about `seconds` of CPU time
    r = int(max(1, min(g.M, seconds / max(t1, 1e-6))))
    t0 = time.perf_counter()
    fn(A, B, g.transA, g.transB, g.alpha, g.beta, C0, pairs=rows_pairs(r))
    dt = time.perf_counter() - t0
    flops = 2.0 * r * g.N * g.K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{r} of {g.M} rows x all {g.N} columns of {g.name} ({g.mode}), "
                      f"{dt:.1f} s, scaled linearly"}


# ------------------------------------------------------- reference arm --

def bench_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    from fp32_emulated_gemm_split_gb300 import workloads as W
    import oracle
    g = pick_workload(W, args)
    A, B, C0 = W.generate(g)
    oracle.build()
    fn = ORACLE_FN(oracle)[g.mode]
    # each step is a block of rows sized so the whole run takes a few minutes
    budget = max(20.0, min(150.0, args.cpu_seconds * 6))
    per_step = budget / (args.steps + args.warmup)
    mi = np.zeros(g.N, np.int64)
    ni = np.arange(g.N, dtype=np.int64)
    t0 = time.perf_counter()
    fn(A, B, g.transA, g.transB, g.alpha, g.beta, C0, pairs=(mi, ni))
    t_row = time.perf_counter() - t0
    rows = int(max(1, min(g.M, per_step / max(t_row, 1e-6))))
    pairs = (np.repeat(np.arange(rows, dtype=np.int64), g.N),
             np.tile(np.arange(g.N, dtype=np.int64), rows))
    for _ in range(args.warmup):
        fn(A, B, g.transA, g.transB, g.alpha, g.beta, C0, pairs=pairs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn(A, B, g.transA, g.transB, g.alpha, g.beta, C0, pairs=pairs)
    dt = (time.perf_counter() - t0) / args.steps
    value = 2.0 * rows * g.N * g.K / dt / 1e12
    sample = f"{rows} of {g.M} rows x all {g.N} columns of {g.name} per step, scaled linearly"
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": g.name, "M": g.M, "N": g.N, "K": g.K, "mode": g.mode,
                   "transA": g.transA, "transB": g.transB, "alpha": g.alpha, "beta": g.beta,
                   "emulates": "fp32"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="square8192_normal")
    ap.add_argument("--mode", default=None,
                    choices=[None, "bf16x9", "tf32x3", "tf32x3_oy", "bf16x3", "tf32", "fp32_simt"])
    ap.add_argument("--impl", default="emu", choices=["emu", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-simt", action="store_true", help="skip the SIMT FP32 context number")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the timing of the other configurations, the accuracy ladder "
                         "and the weight gradients")
    ap.add_argument("--shape", default=None, help="M,N,K override (same distribution)")
    ap.add_argument("--path", default=None, choices=[None, "auto", "twopass", "fused", "fused_tmem"],
                    help="implementation of the tensor-core modes (default: the library's)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)      # at least 3 untimed warm-up steps
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_gpu(args)


if __name__ == "__main__":
    main()

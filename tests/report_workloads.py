"""Accuracy and speed of every workload and mode on the GPU (a report, not a
test): one JSON line per (workload, mode) with

  tflops        effective 2MNK/t of emu_sgemm, one call at a time (CUDA events
                around each call, median of runs: includes the launch latency)
  tflops_stream the same for calls issued back to back (events around a run
                of calls: the host's launch work overlaps the GPU's, as when
                a model runs its layers one after another)
  pct_p9        that figure as a percentage of the measured BF16 peak / 9
  max_ratio     max |C - C_ref| / bound over the checked outputs (<= 1 passes)
  rel_frob      relative Frobenius error over the checked outputs
  checked       "all" or the number of sampled outputs

plus, per workload, the library's SIMT FP32 kernel and, for context, cuBLAS
FP32 through torch.matmul with and without CUBLAS_EMULATE_SINGLE_PRECISION=1
(the cuBLAS BF16x9 path the pages use; run in a child process because cuBLAS
reads the variable when it starts).

  python tests/report_workloads.py [--workloads a,b] [--out file.jsonl] [--no-cublas]
"""
import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
sys.path.insert(0, ROOT)
sys.path.insert(0, HERE)

import oracle  # noqa: E402
from oracle import checks  # noqa: E402
from fp32_emulated_gemm_split_gb300 import workloads as W  # noqa: E402


def time_call(fn, reps=10, warm=3):
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        torch.cuda.synchronize()
        times.append(s.elapsed_time(e))
    return float(np.median(times))


def time_stream(fn, reps=20, rounds=3):
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(rounds):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            fn()
        e.record()
        torch.cuda.synchronize()
        times.append(s.elapsed_time(e) / reps)
    return float(np.median(times))


def cublas_child(name, emulate):
    """Time torch.matmul FP32 on the workload in a child process."""
    code = f"""
import sys, json, torch, numpy as np
sys.path.insert(0, {ROOT!r})
torch.backends.cuda.matmul.allow_tf32 = False
from fp32_emulated_gemm_split_gb300 import workloads as W
g = W.WORKLOADS[{name!r}]
A, B, C0 = W.generate(g)
a = torch.from_numpy(A).cuda(); b = torch.from_numpy(B).cuda()
a = a.t() if g.transA else a
b = b.t() if g.transB else b
f = lambda: torch.matmul(a, b)
for _ in range(3): f()
torch.cuda.synchronize()
ts = []
for _ in range(10):
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(); f(); e.record(); torch.cuda.synchronize(); ts.append(s.elapsed_time(e))
reps = 20 if g.flops < 2e12 else 5
tb = []
for _ in range(3):
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps): f()
    e.record(); torch.cuda.synchronize(); tb.append(s.elapsed_time(e) / reps)
print(json.dumps({{"ms": float(np.median(ts)), "ms_stream": float(np.median(tb))}}))
"""
    env = dict(os.environ)
    if emulate:
        env["CUBLAS_EMULATE_SINGLE_PRECISION"] = "1"
        env["CUBLAS_EMULATION_STRATEGY"] = "eager"
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=600)
    if r.returncode != 0:
        return None, None
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return d["ms"], d["ms_stream"]


def cpu_oracle_time(g, A, B, C0, seconds):
    """The oracle's BF16x9 (plain C, OpenMP over the host cores) on whole rows
    of C: one row to calibrate, then a block of rows sized to `seconds`;
    the whole GEMM's time is extrapolated linearly in rows."""
    import numpy as np

    def rows(r, fn=oracle.gemm_bf16x9):
        mi = np.repeat(np.arange(r, dtype=np.int64), g.N)
        ni = np.tile(np.arange(g.N, dtype=np.int64), r)
        t = time.perf_counter()
        fn(A, B, g.transA, g.transB, g.alpha, g.beta, C0, pairs=(mi, ni))
        return time.perf_counter() - t

    r, t = 1, rows(1)
    for _ in range(3):          # thread start-up makes one row a poor guess
        if t >= seconds / 2 or r >= g.M:
            break
        r = int(max(1, min(g.M, r * seconds / max(t, 1e-6))))
        t = rows(r)
    full = t * g.M / r
    ref_full = rows(r, oracle.gemm_ref) * g.M / r      # the FP64 reference on the same rows
    return {"workload": g.name, "mode": "cpu_oracle_bf16x9", "rows_timed": r,
            "seconds_timed": round(t, 3), "seconds_full": round(full, 3),
            "seconds_full_fp64_ref": round(ref_full, 3),
            "extrapolated": r < g.M, "threads": oracle.max_threads(),
            "tflops": round(g.flops / full / 1e12, 7)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workloads", default=",".join(n for n in W.WORKLOADS if not n.endswith("_tf32x3")))
    ap.add_argument("--out", default=None)
    ap.add_argument("--no-cublas", action="store_true")
    ap.add_argument("--samples", type=int, default=4096)
    ap.add_argument("--cpu-seconds", type=float, default=0.0,
                    help="also time the CPU oracle's BF16x9 on a block of rows of about "
                         "this many seconds per workload and extrapolate to the whole GEMM")
    args = ap.parse_args()

    import torch
    import fp32_emulated_gemm_split_gb300 as emu
    torch.cuda.set_device(0)
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {"bf16_tflops": 1900.0}
    p9 = peaks["bf16_tflops"] / 9.0
    out = open(args.out, "a") if args.out else None

    for name in args.workloads.split(","):
        g0 = W.WORKLOADS[name]
        A, B, C0 = W.generate(g0)
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        full = g0.M * g0.N * g0.K <= 4e9
        if full:
            Cref, Sabs = oracle.gemm_ref(A, B, g0.transA, g0.transB, g0.alpha, g0.beta, C0)
            mi = ni = None
        else:
            mi, ni = W.sample_pairs(g0.M, g0.N, args.samples)
            Cref, Sabs = oracle.gemm_ref(A, B, g0.transA, g0.transB, g0.alpha, g0.beta, C0,
                                         pairs=(mi, ni))
        modes = ["bf16x9", "bf16x9_fused", "bf16x9_fused_tmem", "tf32x3", "tf32x3_oy", "bf16x3",
                 "tf32", "fp32_simt"]
        for mode_name in modes:
            mode, _, path = mode_name.partition("_") if mode_name.startswith("bf16x9_") else (mode_name, "", "")
            emu.emu_set_path(path or "twopass")
            dC = torch.from_numpy(C0).cuda() if C0 is not None else torch.empty((g0.M, g0.N), device="cuda")
            dC0 = dC.clone() if C0 is not None else None

            def run():
                if dC0 is not None:
                    dC.copy_(dC0)
                emu.emu_sgemm(dA, dB, dC, transA=g0.transA, transB=g0.transB, alpha=g0.alpha,
                              beta=g0.beta, mode=mode)

            run()
            torch.cuda.synchronize()
            if full:
                got = dC.cpu().numpy()
                C0s = C0
            else:
                got = dC[torch.from_numpy(mi).cuda(), torch.from_numpy(ni).cuda()].cpu().numpy()
                C0s = C0[mi, ni] if C0 is not None else None
            bmode = mode if mode in checks.MODE_EXTRA else "bf16x9"
            ratio = checks.error_ratio(got, Cref, Sabs, g0.K, g0.alpha, g0.beta, C0s, mode=bmode)
            relf = checks.rel_frobenius(got, Cref)
            reps = 10 if g0.flops < 2e12 else 5
            ms = time_call(run, reps=reps)
            ms_s = time_stream(run, reps=2 * reps)
            if dC0 is not None:   # subtract the restore copy of C
                ms -= time_call(lambda: dC.copy_(dC0), reps=reps)
                ms_s -= time_stream(lambda: dC.copy_(dC0), reps=2 * reps)
            tf = g0.flops / (ms * 1e-3) / 1e12
            tfs = g0.flops / (ms_s * 1e-3) / 1e12
            rec = {"workload": name, "mode": mode_name, "M": g0.M, "N": g0.N, "K": g0.K,
                   "ms": round(ms, 4), "tflops": round(tf, 2), "pct_p9": round(100 * tf / p9, 1),
                   "ms_stream": round(ms_s, 4), "tflops_stream": round(tfs, 2),
                   "pct_p9_stream": round(100 * tfs / p9, 1),
                   "max_ratio": ratio, "rel_frob": relf,
                   "checked": "all" if full else int(mi.size)}
            print(json.dumps(rec), flush=True)
            if out:
                out.write(json.dumps(rec) + "\n")
        emu.emu_set_path("auto")
        if not args.no_cublas and g0.mode == "bf16x9":
            for emulate in (False, True):
                ms, ms_s = cublas_child(name, emulate)
                rec = {"workload": name, "mode": "cublas_" + ("bf16x9_env" if emulate else "fp32"),
                       "ms": ms, "tflops": None if ms is None else round(g0.flops / (ms * 1e-3) / 1e12, 2),
                       "ms_stream": ms_s,
                       "tflops_stream": None if ms_s is None else round(g0.flops / (ms_s * 1e-3) / 1e12, 2)}
                print(json.dumps(rec), flush=True)
                if out:
                    out.write(json.dumps(rec) + "\n")
        if args.cpu_seconds > 0:
            rec = cpu_oracle_time(g0, A, B, C0, args.cpu_seconds)
            print(json.dumps(rec), flush=True)
            if out:
                out.write(json.dumps(rec) + "\n")
        del dA, dB
        torch.cuda.empty_cache()
    assert emu.emu_get_last_device_error() == 0


if __name__ == "__main__":
    main()

"""Time emu_sgemm per call over a grid of shapes, in each tensor-core mode and
with the FP32 SIMT kernel, on the GPU (a measurement, not a test): the data
behind the PERFORMANT strategy's choice between emulation and plain FP32.

For every (M, N, K) it prints one JSON line with, per mode, the device time
of one call measured two ways after warm-up:
  eager_us  CUDA events around R back-to-back calls from Python, divided by
            R (host overhead included when the host is the bottleneck);
  graph_us  the same R calls captured in a CUDA graph and replayed (device
            time, launch gaps included, host overhead excluded).
The library is forced to the EAGER strategy so each mode runs as asked.

  python tests/chooser_sweep.py [--out file.jsonl] [--reps 20]
"""
import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

SIZES_MN = [64, 256, 1024, 4096]
SIZES_K = [16, 64, 256, 1024, 4096]
EXTRA = [(12288, 256, 256), (12288, 1024, 256), (12288, 256, 1024), (256, 12288, 256),
         (8192, 8192, 64), (2048, 2048, 2048)]
MODES = ["bf16x9", "tf32x3", "fp32_simt"]


def time_mode(emu, torch, A, B, C, mode, reps):
    def call():
        emu.emu_sgemm(A, B, C, mode=mode)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        call()
    e.record()
    e.synchronize()
    eager = s.elapsed_time(e) * 1e3 / reps
    graph = None
    try:
        st = torch.cuda.Stream()
        with torch.cuda.stream(st):
            call()                       # workspace sized before the capture
            st.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                for _ in range(reps):
                    emu.emu_sgemm(A, B, C, mode=mode, stream=st)
            g.replay()
            st.synchronize()
            s.record(st)
            g.replay()
            e.record(st)
            e.synchronize()
        graph = s.elapsed_time(e) * 1e3 / reps
    except Exception as ex:              # report, keep sweeping
        graph = f"capture failed: {ex}"
    return round(eager, 2), graph if isinstance(graph, str) else round(graph, 2)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=None)
    ap.add_argument("--reps", type=int, default=20)
    args = ap.parse_args()
    import torch
    import fp32_emulated_gemm_split_gb300 as emu
    emu.emu_set_strategy("eager")
    shapes = [(m, n, k) for m in SIZES_MN for n in SIZES_MN for k in SIZES_K] + EXTRA
    out = open(args.out, "a") if args.out else None
    gen = torch.Generator(device="cuda").manual_seed(3)
    for (M, N, K) in shapes:
        A = torch.randn((M, K), device="cuda", generator=gen)
        B = torch.randn((K, N), device="cuda", generator=gen)
        C = torch.empty((M, N), device="cuda")
        rec = {"M": M, "N": N, "K": K}
        for mode in MODES:
            eager, graph = time_mode(emu, torch, A, B, C, mode, args.reps)
            rec[mode] = {"eager_us": eager, "graph_us": graph}
        rec["choice"] = emu.emu_choose_mode(M, N, K, "bf16x9", strategy="performant")
        print(json.dumps(rec), flush=True)
        if out:
            out.write(json.dumps(rec) + "\n")
    assert emu.emu_get_last_device_error() == 0


if __name__ == "__main__":
    main()

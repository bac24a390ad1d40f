"""Measure g_predict for every micro-kernel of the set (offline, once per machine).

The MikPoly summary (section 3, "micro-kernel performance model") pre-runs each
micro-kernel for pipeline tasks of t = 1..T micro-kernel instances and keeps the
times as g_predict(t).  Here each micro-kernel is forced (mp_force_plan, no
split-K) onto a GEMM whose tiles fill exactly one wave of the GPU, at several K
= t * 64, and timed back to back with CUDA events; a least-squares line

    g_predict(t) = fixed_us + per_step_us * t

is fitted per micro-kernel (the persistent kernel runs one task per SM, so a
one-wave launch time is the time of one pipeline task under full-wave load,
launch and epilogue included).  The table is written in the text format that
mp_init reads ("um un uk swap fixed_us per_step_us").

    python -m micro_polymerization_gb300.calibrate [--out PATH] [--device 0]
"""
from __future__ import annotations

import argparse
import os
import sys

DEFAULT_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "calib", "gb300.txt")
STEPS = (2, 8, 32, 96)


def one_wave_shape(desc, hw):
    """(M, N) whose tiles of this micro-kernel fill one wave of its task slots
    (warps_per_wave / warps: one task per SM, or per SM pair for pair kernels)."""
    slots = max(1, hw.warps_per_wave // max(1, desc.warps))
    tn = 8 if not desc.swap else 6
    while tn > 1 and slots % tn:
        tn -= 1
    tm = max(1, slots // tn)
    return tm * desc.um, tn * desc.un


def measure(device: int = 0, reps: int = 30):
    import torch
    import micro_polymerization_gb300 as mp
    from micro_polymerization_gb300 import workloads as wl

    dev = torch.device("cuda", device)
    torch.cuda.set_device(dev)
    h = mp.mp_init(device)
    hw, kernels = mp.mp_get_hw(h)
    lib = mp.library()
    sp = torch.cuda.current_stream().cuda_stream
    rows = []
    try:
        for k, desc in enumerate(kernels):
            mp.mp_force_plan(h, k, 1)
            M, N = one_wave_shape(desc, hw)
            pts = []
            for t in STEPS:
                K = 64 * t
                A, B, _ = wl.make_operands(wl.Gemm(M, N, K, seed=5), device=dev)
                D = torch.empty(M, N, device=dev)
                args = (h.ptr, M, N, K, A.data_ptr(), K, B.data_ptr(), N, None, N, D.data_ptr(), N, 1.0, 0.0, sp)
                for _ in range(5):
                    lib.mp_gemm(*args)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record()
                for _ in range(reps):
                    st = lib.mp_gemm(*args)
                    if st != 0:
                        raise mp.MPError(st, "mp_gemm")
                e1.record()
                torch.cuda.synchronize()
                pts.append((t, e0.elapsed_time(e1) * 1e3 / reps))
            n = len(pts)
            sx = sum(t for t, _ in pts)
            sy = sum(y for _, y in pts)
            sxx = sum(t * t for t, _ in pts)
            sxy = sum(t * y for t, y in pts)
            slope = (n * sxy - sx * sy) / (n * sxx - sx * sx)
            icpt = (sy - slope * sx) / n
            rows.append((desc, max(0.0, icpt), max(1e-3, slope), pts, (M, N)))
    finally:
        mp.mp_force_plan(h, -1, 0)
        h.close()
    return hw, rows


def write_table(path: str, hw, rows) -> None:
    os.makedirs(os.path.dirname(path), exist_ok=True)
    with open(path, "w") as f:
        f.write("# g_predict(t) = fixed_us + per_step_us * t per micro-kernel, measured on one GPU with\n")
        f.write(f"# {hw.num_pe} SMs by micro_polymerization_gb300/calibrate.py: one wave of tiles, K = 64 t,\n")
        f.write(f"# t in {STEPS}, back-to-back CUDA-event times, least-squares line.\n")
        f.write("# um un uk swap fixed_us per_step_us   # one-wave shape (M, N): measured (t, us)\n")
        for desc, icpt, slope, pts, (M, N) in rows:
            meas = " ".join(f"({t},{y:.2f})" for t, y in pts)
            f.write(f"{desc.um} {desc.un} {desc.uk} {desc.swap} {icpt:.4f} {slope:.5f}   # ({M},{N}): {meas}\n")


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--out", default=DEFAULT_PATH)
    ap.add_argument("--device", type=int, default=0)
    args = ap.parse_args(argv)
    hw, rows = measure(args.device)
    write_table(args.out, hw, rows)
    with open(args.out) as f:
        sys.stdout.write(f.read())
    return 0


if __name__ == "__main__":
    sys.exit(main())

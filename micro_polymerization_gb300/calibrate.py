"""Measure g_predict for every micro-kernel of the set (offline, once per machine).

The MikPoly summary (section 3, "micro-kernel performance model") pre-runs each
micro-kernel for pipeline tasks of t = 1..T micro-kernel instances and keeps the
times as g_predict(t).  Each micro-kernel here is forced (mp_force_plan, no
split-K) onto GEMMs whose tiles fill exactly one wave and exactly two waves of
its task slots, at K = 64 t for several t.  Every time is device time per call
of calls made back to back through the C ABI, cycling over copies of the
operands that together exceed twice L2, so that operands arrive cold from HBM
as in the dynamic-shape workloads.  Two forms of table can be written, in the
text format mp_init reads ("um un uk swap fixed_us per_step_us tail_us"):

  one-wave (default): g_predict(t) = fixed_us + per_step_us * t is the
      least-squares line through the one-wave times; launch, pipeline fill and
      the write-back are inside fixed_us, charged in every task, and tail_us
      is 0 -- the structure of the analytic default model;
  waves: the section's three overlapped stages taken at their word (a task's
      write-back hidden behind the next task on the same PE): g_predict(t) is
      the line through the two-wave minus one-wave times and tail_us, charged
      once per plan, the rest of the one-wave time.

Measured on GB300 the second wave costs its K loop plus most of an epilogue
(the first wave's stores slow the second wave's operand loads), and planning
with the "waves" form made the dynamic-shape steps 1-7% slower.

    python -m micro_polymerization_gb300.calibrate [--out PATH] [--device 0] [--form one-wave|waves]

With --form one-wave (the default) the table holds the least-squares line
through the one-wave times alone (launch, fill and the write-back inside
fixed_us, tail 0): the structure of the analytic default model.
"""
from __future__ import annotations

import argparse
import math
import os
import sys

DEFAULT_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "calib", "gb300.txt")
STEPS = (4, 12, 24)
L2_BYTES = 126 * 2 ** 20


def wave_shape(desc, hw, waves):
    """(M, N) whose tiles of this micro-kernel fill `waves` waves of its task
    slots (warps_per_wave / warps: one task per SM, or per SM pair for pair
    kernels)."""
    slots = max(1, hw.warps_per_wave // max(1, desc.warps))
    tn = 8 if not desc.swap else 6
    while tn > 1 and slots % tn:
        tn -= 1
    tm = max(1, slots // tn) * waves
    return tm * desc.um, tn * desc.un


def time_cold(lib, h, M, N, K, sp, reps=3):
    """Device time (us) per back-to-back call of one GEMM, operands cold."""
    import torch
    from micro_polymerization_gb300 import workloads as wl
    import micro_polymerization_gb300 as mp
    dev = torch.device("cuda", torch.cuda.current_device())
    A, B, _ = wl.make_operands(wl.Gemm(M, N, K, seed=5), device=dev)
    D = torch.empty(M, N, device=dev)
    nbytes = 2 * (M * K + K * N) + 4 * M * N
    copies = int(min(32, max(2, math.ceil(2 * L2_BYTES / nbytes))))
    sets = [(A, B, D)] + [(A.clone(), B.clone(), torch.empty_like(D)) for _ in range(copies - 1)]
    calls = [(h.ptr, M, N, K, a.data_ptr(), K, b.data_ptr(), N, None, N, d.data_ptr(), N, 1.0, 0.0, sp)
             for a, b, d in sets]

    def run():
        for c in calls:
            st = lib.mp_gemm(*c)
            if st != 0:
                raise mp.MPError(st, "mp_gemm")

    run()
    best = float("inf")
    for _ in range(reps):
        torch.cuda._sleep(20_000_000)  # hold the GPU while the calls are queued
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1e3 / len(calls))
    return best


def measure(device: int = 0):
    import torch
    import micro_polymerization_gb300 as mp

    torch.cuda.set_device(device)
    h = mp.mp_init(device)
    hw, kernels = mp.mp_get_hw(h)
    lib = mp.library()
    sp = torch.cuda.current_stream().cuda_stream
    rows = []
    try:
        for k, desc in enumerate(kernels):
            mp.mp_force_plan(h, k, 1)
            (M1, N1), (M2, N2) = wave_shape(desc, hw, 1), wave_shape(desc, hw, 2)
            pts = []
            for t in STEPS:
                K = 64 * t
                pts.append((t, time_cold(lib, h, M1, N1, K, sp), time_cold(lib, h, M2, N2, K, sp)))
            # g_predict(t) = T2(t) - T1(t): least-squares line in t.
            n = len(pts)
            xs = [t for t, _, _ in pts]
            ys = [t2 - t1 for _, t1, t2 in pts]
            sx, sy = sum(xs), sum(ys)
            sxx = sum(x * x for x in xs)
            sxy = sum(x * y for x, y in zip(xs, ys))
            slope = (n * sxy - sx * sy) / (n * sxx - sx * sx)
            icpt = (sy - slope * sx) / n
            fixed, step = max(0.0, icpt), max(1e-3, slope)
            tail = max(0.0, sum(t1 - (fixed + step * t) for t, t1, _ in pts) / n)
            # The line through the one-wave times alone (launch, fill and the
            # write-back inside its intercept).
            y1 = [t1 for _, t1, _ in pts]
            s1y, s1xy = sum(y1), sum(x * y for x, y in zip(xs, y1))
            slope1 = (n * s1xy - sx * s1y) / (n * sxx - sx * sx)
            icpt1 = (s1y - slope1 * sx) / n
            rows.append((desc, fixed, step, tail, max(0.0, icpt1), max(1e-3, slope1), pts, (M1, N1), (M2, N2)))
    finally:
        mp.mp_force_plan(h, -1, 0)
        h.close()
    return hw, rows


def write_table(path: str, hw, rows, form: str = "one-wave") -> None:
    """form "one-wave": g_predict is the line through the one-wave times
    (tail 0); "waves": g_predict is the two-wave minus one-wave line and the
    rest of the one-wave time is the tail."""
    os.makedirs(os.path.dirname(path), exist_ok=True)
    with open(path, "w") as f:
        f.write("# g_predict(t) = fixed_us + per_step_us * t and tail_us per micro-kernel, measured on one GPU\n")
        f.write(f"# with {hw.num_pe} SMs by micro_polymerization_gb300/calibrate.py (form {form}): one and two\n")
        f.write(f"# waves of tiles, K = 64 t, t in {STEPS}, device time per back-to-back call on cold operands.\n")
        f.write("# um un uk swap fixed_us per_step_us tail_us   # one- and two-wave (M, N): (t, T1, T2) in us\n")
        for desc, fixed, step, tail, fixed1, step1, pts, s1, s2 in rows:
            if form == "one-wave":
                fixed, step, tail = fixed1, step1, 0.0
            meas = " ".join(f"({t},{a:.2f},{b:.2f})" for t, a, b in pts)
            f.write(f"{desc.um} {desc.un} {desc.uk} {desc.swap} {fixed:.4f} {step:.5f} {tail:.4f}"
                    f"   # {s1} {s2}: {meas}\n")


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--out", default=DEFAULT_PATH)
    ap.add_argument("--device", type=int, default=0)
    ap.add_argument("--form", choices=["one-wave", "waves"], default="one-wave")
    args = ap.parse_args(argv)
    hw, rows = measure(args.device)
    write_table(args.out, hw, rows, args.form)
    with open(args.out) as f:
        sys.stdout.write(f.read())
    return 0


if __name__ == "__main__":
    sys.exit(main())

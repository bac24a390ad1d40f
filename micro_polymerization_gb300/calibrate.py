"""Measure g_predict for every micro-kernel of the set (offline, once per machine).

The MikPoly summary (section 3, "micro-kernel performance model") pre-runs each
micro-kernel for pipeline tasks of t = 1..T micro-kernel instances and keeps the
times as g_predict(t).  Each micro-kernel here is forced (mp_force_plan, no
split-K) onto GEMMs whose tiles fill exactly one wave and exactly two waves of
its task slots, at K = 64 t for several t.  Every time is the device time a
call adds to a stream of different GEMMs, as in the dynamic-shape workloads:
the calls alternate with calls of a fixed reference GEMM, both cycling over
copies of their operands that exceed twice L2 (operands arrive cold from
HBM), and the reference's own time is subtracted.  Back-to-back calls of one
shape (--back-to-back) hide what a launch with thread-block clusters costs
after a different kernel: 1-6 us on GB300 for CTA pairs and split-K on chip.
Two forms of table can be written, in the text format mp_init reads
("um un uk swap fixed_us per_step_us tail_us"):

  waves (default): the section's three overlapped stages -- a wave's
      write-back hides behind the next wave's tasks on the same PEs: a
      plan's first wave costs the one-wave line (launch, pipeline fill, the
      K steps, the last write-back and what a cluster launch costs after a
      different kernel), and every further wave what a second wave was
      measured to add beyond its K steps, plus the one-wave rate per K step.
      In the table: fixed_us that per-wave term, per_step_us the one-wave
      slope, tail_us (charged once per plan) the rest of the one-wave
      intercept;
  one-wave: the least-squares line through the one-wave times; launch, fill
      and the write-back are inside fixed_us, charged in every wave, and
      tail_us is 0 -- the structure of the analytic model.

Measured on GB300 against the analytic model (bench.py, the same box, three
runs each, two calibrations on two boxes): waves tables timed in the mixed
stream planned the dynamic-sequence step 0.3-0.8% faster, dynamic resolution
0.4-0.5% and merged QKV 0.6-0.9% faster, the batched merge 0-1.5% slower and
the skinny GEMM even.  On the stress sweep (alpha 1.5, beta 0.5) the table
planned 1.7% slower: it is calibrated with beta = 0, and with beta * C a
partly filled 128-row tile's epilogue leaves most of its warps idle, where
the swapped tiles the analytic model picks for small M do not.  Charging
later waves the two-wave increment's own slope instead let one-wave CTA-pair
plans of (3520..4032, 768, 3072) look cheap and made the step 3% slower; the
one-wave form charges a pair's launch cost in every wave and moved a 29-wave
GEMM of the stress sample off CTA pairs; tables timed back to back made the
steps 1-7% slower.

The split-K reduction is measured the same way: one-CTA micro-kernels forced
to split K S ways (S = 2..8 reduce on chip in clusters of S CTAs; S = 12, 16
through L2) on one wave of tasks, K = 64 t S.  What a call costs beyond the
kernel's own one-wave line at f_num = t is the reduction; the least-squares
fit of it against the tile's fp32 bytes at one PE's share of L2 gives the
table's "split on_chip sync_us bytes_factor [S]" lines: one per cluster size
on chip (the on-chip sum costs more at S = 2 and 3 than at 4 to 8), one
through L2.

    python -m micro_polymerization_gb300.calibrate [--out PATH] [--device 0] [--form waves|one-wave]
                                                    [--back-to-back]

The default --out is the table mp_init loads by default (calib/gb300.txt).
"""
from __future__ import annotations

import argparse
import math
import os
import sys

DEFAULT_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "calib", "gb300.txt")
STEPS = (4, 12, 24)
SPLIT_STEPS = (4, 12)
SPLIT_ON_CHIP = (2, 3, 4, 5, 6, 7, 8)   # cluster sizes, each fitted apart
SPLIT_THROUGH_L2 = (12, 16)
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


# The reference GEMM of the mixed stream: one wave of 128 x 256 one-CTA tiles
# (the first micro-kernel of the set, forced), K = 768.
REF_SHAPE = (2048, 2304, 768)
REF_PAIRS = 32


class Mixed:
    """Times a GEMM as its marginal cost in a stream of different GEMMs: its
    calls alternate with calls of a fixed reference GEMM, and the reference's
    own time (its calls back to back) is subtracted.  Measured on GB300, a
    launch that uses thread-block clusters (CTA pairs, split-K on chip) costs
    1-6 us more after a different kernel than after a copy of itself, which
    back-to-back calls of one shape never show; a dynamic-shape workload is
    such a stream."""

    def __init__(self, lib, sp, device):
        import micro_polymerization_gb300 as mp
        self.lib, self.sp = lib, sp
        self.h = mp.mp_init(device)
        mp.mp_force_plan(self.h, 0, 1)
        self.calls = None
        self.t_ref = None

    def ref_calls(self):
        """REF_PAIRS calls of the reference GEMM on their own operand copies
        (together twice L2), timed back to back once (t_ref, us per call)."""
        import torch
        from micro_polymerization_gb300 import workloads as wl
        if self.calls is None:
            M, N, K = REF_SHAPE
            dev = torch.device("cuda", torch.cuda.current_device())
            A, B, _ = wl.make_operands(wl.Gemm(M, N, K, seed=11), device=dev)
            self.sets = [(A.clone(), B.clone(), torch.empty(M, N, device=dev)) for _ in range(REF_PAIRS)]
            self.calls = [(self.h.ptr, M, N, K, a.data_ptr(), K, b.data_ptr(), N, None, N, d.data_ptr(), N, 1.0, 0.0,
                           self.sp) for a, b, d in self.sets]
            self.t_ref = run_timed(self.lib, self.calls) / REF_PAIRS
        return self.calls

    def close(self):
        self.h.close()


def run_timed(lib, calls, reps=3):
    """Best device time (us) of one run of `calls`, queued behind a sleep."""
    import torch
    import micro_polymerization_gb300 as mp
    for c in calls:
        st = lib.mp_gemm(*c)
        if st != 0:
            raise mp.MPError(st, "mp_gemm")
    best = float("inf")
    for _ in range(reps):
        torch.cuda._sleep(20_000_000)  # hold the GPU while the calls are queued
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for c in calls:
            lib.mp_gemm(*c)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1e3)
    return best


def time_cold(lib, h, M, N, K, sp, mixed=None, reps=3):
    """Device time (us) per call of one GEMM on cold operands: calls cycle over
    copies of the operands that together exceed twice L2.  With `mixed`
    (a Mixed), the calls alternate with the reference GEMM and the time is the
    marginal cost per call; otherwise the calls run back to back."""
    import torch
    from micro_polymerization_gb300 import workloads as wl
    dev = torch.device("cuda", torch.cuda.current_device())
    A, B, _ = wl.make_operands(wl.Gemm(M, N, K, seed=5), device=dev)
    D = torch.empty(M, N, device=dev)
    nbytes = 2 * (M * K + K * N) + 4 * M * N
    copies = int(min(32, max(2, math.ceil(2 * L2_BYTES / nbytes))))
    sets = [(A, B, D)] + [(A.clone(), B.clone(), torch.empty_like(D)) for _ in range(copies - 1)]
    calls = [(h.ptr, M, N, K, a.data_ptr(), K, b.data_ptr(), N, None, N, d.data_ptr(), N, 1.0, 0.0, sp)
             for a, b, d in sets]
    if mixed is None:
        return run_timed(lib, calls, reps) / len(calls)
    ref = mixed.ref_calls()
    seq = [c for i in range(REF_PAIRS) for c in (ref[i], calls[i % len(calls)])]
    return run_timed(lib, seq, reps) / REF_PAIRS - mixed.t_ref


def split_shape(desc, tiles):
    """(M, N) of `tiles` tiles of a one-CTA micro-kernel in one row (swapped:
    one column) of tiles."""
    if desc.swap:
        return desc.um, tiles * desc.un
    return tiles * desc.um, desc.un


def fit_line(xs, ys):
    """Least-squares (intercept, slope >= 0) of ys against xs."""
    n = len(xs)
    sx, sy = sum(xs), sum(ys)
    sxx = sum(x * x for x in xs)
    sxy = sum(x * y for x, y in zip(xs, ys))
    den = n * sxx - sx * sx
    slope = (n * sxy - sx * sy) / den if den > 0 else 0.0
    if slope < 0:
        slope = 0.0
    return max(0.0, (sy - slope * sx) / n), slope


def fit_kernel(pts):
    """(fixed_us, per_step_us, tail_us, fixed1_us, step1_us) from one
    micro-kernel's (t, T1, T2) points.  fixed1 + step1 t is the least-squares
    line through the one-wave times.  The waves form charges a plan's first
    wave that line and every further wave the intercept of the two-wave minus
    one-wave line (what one more wave adds beyond its K steps: mostly the
    write-back the next wave does not hide) plus step1 per K step; the rest of
    the one-wave intercept is the tail, once per plan.  The two-wave increment
    steps faster than one wave alone (the calibration's second wave finds its
    B columns in L2); charging every wave the one-wave slope planned the
    measured steps better."""
    xs = [t for t, _, _ in pts]
    fixed_w, _ = fit_line(xs, [t2 - t1 for _, t1, t2 in pts])
    fixed1, step1 = fit_line(xs, [t1 for _, t1, _ in pts])
    step1 = max(1e-3, step1)
    return fixed_w, step1, max(0.0, fixed1 - fixed_w), fixed1, step1


def measure_split(lib, h, hw, kernels, lines, sp, mixed=None):
    """Split-K overhead per call beyond each kernel's one-wave line, fitted
    per reduction path: key 0 through L2, key S on chip in clusters of S.
    lines: kernel index -> (fixed_us, per_step_us)."""
    import micro_polymerization_gb300 as mp
    slots = max(1, hw.warps_per_wave // max(1, kernels[0].warps))
    pe_gbs = hw.l2_gbs / max(1, hw.num_pe)
    groups = [(S, (S,), True) for S in SPLIT_ON_CHIP] + [(0, SPLIT_THROUGH_L2, False)]
    out = {}
    try:
        for key, Ss, on_chip in groups:
            xs, ys, pts = [], [], []
            for k, desc in enumerate(kernels):
                if desc.pair or k not in lines:
                    continue
                fixed, step = lines[k]
                x = 4.0 * desc.um * desc.un / (pe_gbs * 1e3)  # one pass over the fp32 partial, us
                for S in Ss:
                    # On chip: at most 96 tasks, which every cluster size up to
                    # 8 keeps resident on one GB300; through L2: one wave.
                    tiles = max(1, (96 if on_chip else slots) // S)
                    M, N = split_shape(desc, tiles)
                    mp.mp_force_plan(h, k, S)
                    for t in SPLIT_STEPS:
                        T = time_cold(lib, h, M, N, 64 * t * S, sp, mixed)
                        xs.append(x)
                        ys.append(T - (fixed + step * t))
                        pts.append((desc.um, desc.un, desc.swap, S, t, round(T, 2)))
            out[key] = fit_line(xs, ys) + (pts,)
    finally:
        mp.mp_force_plan(h, -1, 0)
    return out


def measure(device: int = 0, back_to_back: bool = False):
    import torch
    import micro_polymerization_gb300 as mp

    torch.cuda.set_device(device)
    h = mp.mp_init(device)
    hw, kernels = mp.mp_get_hw(h)
    lib = mp.library()
    sp = torch.cuda.current_stream().cuda_stream
    mixed = None if back_to_back else Mixed(lib, sp, device)
    rows = []
    try:
        for k, desc in enumerate(kernels):
            mp.mp_force_plan(h, k, 1)
            (M1, N1), (M2, N2) = wave_shape(desc, hw, 1), wave_shape(desc, hw, 2)
            pts = []
            for t in STEPS:
                K = 64 * t
                pts.append((t, time_cold(lib, h, M1, N1, K, sp, mixed), time_cold(lib, h, M2, N2, K, sp, mixed)))
            rows.append((desc,) + fit_kernel(pts) + (pts, (M1, N1), (M2, N2)))
        lines = {k: (r[4], r[5]) for k, r in enumerate(rows)}
        split = measure_split(lib, h, hw, kernels, lines, sp, mixed)
    finally:
        mp.mp_force_plan(h, -1, 0)
        h.close()
        if mixed is not None:
            mixed.close()
    return hw, rows, split


def write_table(path: str, hw, rows, form: str = "waves", split=None, mixed: bool = True) -> None:
    """form "one-wave": g_predict is the line through the one-wave times
    (tail 0); "waves": g_predict is the two-wave minus one-wave line and the
    rest of the one-wave time is the tail.  split: key -> (sync_us,
    bytes_factor, points), key 0 through L2 and S on chip, written as
    "split" lines (the split overhead is measured against the one-wave
    lines)."""
    os.makedirs(os.path.dirname(path), exist_ok=True)
    with open(path, "w") as f:
        f.write("# g_predict(t) = fixed_us + per_step_us * t and tail_us per micro-kernel, measured on one GPU\n")
        f.write(f"# with {hw.num_pe} SMs by micro_polymerization_gb300/calibrate.py (form {form}): one and two\n")
        how = ("device time a call adds to a stream alternating with a reference GEMM" if mixed
               else "device time per back-to-back call")
        f.write(f"# waves of tiles, K = 64 t, t in {STEPS}; {how}, cold operands.\n")
        f.write("# um un uk swap fixed_us per_step_us tail_us   # one- and two-wave (M, N): (t, T1, T2) in us\n")
        for desc, fixed, step, tail, fixed1, step1, pts, s1, s2 in rows:
            if form == "one-wave":
                fixed, step, tail = fixed1, step1, 0.0
            meas = " ".join(f"({t},{a:.2f},{b:.2f})" for t, a, b in pts)
            f.write(f"{desc.um} {desc.un} {desc.uk} {desc.swap} {fixed:.4f} {step:.5f} {tail:.4f}"
                    f"   # {s1} {s2}: {meas}\n")
        if split:
            f.write("# split on_chip sync_us bytes_factor [S]   # (um, un, swap, S, t, us per call)\n")
            for key in sorted(split):
                sync_us, factor, pts = split[key]
                meas = " ".join(f"({a},{b},{c},{S},{t},{T})" for a, b, c, S, t, T in pts)
                tail = f" {key}" if key else ""
                f.write(f"split {1 if key else 0} {sync_us:.4f} {factor:.4f}{tail}   # {meas}\n")


class _Desc:
    def __init__(self, um, un, uk, swap):
        self.um, self.un, self.uk, self.swap = um, un, uk, swap


class _Hw:
    def __init__(self, num_pe):
        self.num_pe = num_pe


def refit(src: str, out: str, form: str = "waves") -> None:
    """Rewrite a table from the measurements its comments record (each
    micro-kernel's (t, T1, T2) points; the split lines are kept as they are,
    their fit does not depend on the form)."""
    import re
    rows, split, num_pe, mixed = [], {}, 0, True
    num = r"(-?[\d.]+)"
    for line in open(src):
        m = re.search(r"with (\d+) SMs", line)
        if line.startswith("#"):
            if m:
                num_pe = int(m.group(1))
            if "back-to-back" in line:
                mixed = False
            continue
        head, _, com = line.partition("#")
        f = head.split()
        if not f:
            continue
        if f[0] == "split":
            key = int(f[4]) if len(f) > 4 else 0
            pts = [tuple(int(x) for x in g[:5]) + (float(g[5]),)
                   for g in re.findall(r"\((\d+),(\d+),(\d+),(\d+),(\d+),([\d.]+)\)", com)]
            split[key] = (float(f[2]), float(f[3]), pts)
            continue
        shapes = re.findall(r"\((\d+), (\d+)\)", com)
        pts = [(int(a), float(b), float(c)) for a, b, c in re.findall(r"\(" + num + "," + num + "," + num + r"\)", com)]
        if len(pts) < 2 or len(shapes) < 2:
            raise ValueError(f"{src}: no measurements recorded for {' '.join(f[:4])}")
        desc = _Desc(*(int(x) for x in f[:4]))
        rows.append((desc,) + fit_kernel(pts) + (pts, tuple(map(int, shapes[0])), tuple(map(int, shapes[1]))))
    write_table(out, _Hw(num_pe), rows, form, split, mixed)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--out", default=DEFAULT_PATH)
    ap.add_argument("--device", type=int, default=0)
    ap.add_argument("--form", choices=["waves", "one-wave"], default="waves")
    ap.add_argument("--back-to-back", action="store_true",
                    help="time each GEMM's calls back to back instead of in the mixed stream")
    ap.add_argument("--refit", metavar="TABLE", default=None,
                    help="no GPU: rewrite TABLE in --form from the measurements it records")
    args = ap.parse_args(argv)
    if args.refit:
        refit(args.refit, args.out, args.form)
        with open(args.out) as f:
            sys.stdout.write(f.read())
        return 0
    hw, rows, split = measure(args.device, args.back_to_back)
    write_table(args.out, hw, rows, args.form, split, mixed=not args.back_to_back)
    with open(args.out) as f:
        sys.stdout.write(f.read())
    return 0


if __name__ == "__main__":
    sys.exit(main())

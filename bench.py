"""Benchmark: dynamic-shape GEMM throughput (TFLOPS, device-timed, planning
included) and the fraction of each shape's roofline.

One step = the whole hot path over one batch of synthetic input: 64 GEMMs of
the dynamic-sequence-length workload (M = 8 * seq, seq uniform on [1, 512];
(N, K) cycling over a Transformer layer's four projections; beta = 0), each
planned and launched through the C ABI (mp_gemm) back to back on one stream.
Every GEMM has its own operand buffers, 1.4 GB in all -- larger than the
129 MB L2 -- so no operand is still cached when it is read again.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mp|reference]
                    [--workload NAME] [--sweep]

Prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle on a
bounded sample of the same workload instead.  ``--sweep`` also writes one
summary line per workload to stderr.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "dynamic-shape GEMM TFLOPS (device-timed, incl. planning) and % of per-shape roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic of the persistent kernel from one ncu capture of a small case
# (profiles/k_poly_gemm_launches_dynamic_sequence.md), valid only for the
# kernel source it was taken on: dram__bytes_read.sum over the algorithmic
# operand bytes (2MK + 2KN), and dram__bytes_write.sum over the algorithmic
# output bytes (4MN), summed over the captured launches.
TRAFFIC_RECORD = {"kernel_sha1": "c21f5821fc1e5abd8a41498492b6a11965f24b64", "read_per_alg_read": 1.0051,
                  "write_per_alg_write": 0.0}


# --epilogue: (activation, bf16 D) of mp_gemm_ex.
EPILOGUES = {"none": (0, False), "relu": (1, False), "gelu": (2, False), "bf16": (0, True),
             "relu+bf16": (1, True), "gelu+bf16": (2, True)}


CALIB_TABLE = os.path.join(ROOT, "micro_polymerization_gb300", "calib", "gb300.txt")


def calib_arg(args):
    """mp_init's calib_path: the shipped GB300 table ("" -- the analytic model
    -- with --no-calib or when the table is missing)."""
    return CALIB_TABLE if (os.path.exists(CALIB_TABLE) and not args.no_calib) else ""


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"]))}, "measured"
    except Exception:
        return dict(PEAKS_FALLBACK), "fallback"


def traffic_fields(gs, sel, epi):
    """roofline.traffic (DRAM bytes per launch of the selected launches) and
    its read and write parts, from TRAFFIC_RECORD scaled by each launch's
    algorithmic bytes; all null when the record belongs to other kernel
    source."""
    rec = TRAFFIC_RECORD
    ok = rec["kernel_sha1"] == kernel_sha1() and not epi and rec["read_per_alg_read"] is not None
    note = ("dram__bytes_read.sum + dram__bytes_write.sum per launch from one ncu capture, as ratios to the "
            "algorithmic operand bytes (2MK+2KN) and output bytes (4MN), scaled to these launches; much of "
            "D's fp32 write-back leaves L2 after a launch ends, so traffic_write undercounts D")
    if not ok:
        return {"traffic": None, "traffic_read": None, "traffic_write": None,
                "traffic_note": "no ncu record for this kernel source"}
    rd = sum(2.0 * gs[i].M * gs[i].K + 2.0 * gs[i].K * gs[i].N for i in sel) / max(1, len(sel))
    wr = sum(4.0 * gs[i].M * gs[i].N for i in sel) / max(1, len(sel))
    r, w = rec["read_per_alg_read"] * rd, rec["write_per_alg_write"] * wr
    return {"traffic": round(r + w), "traffic_read": round(r), "traffic_write": round(w), "traffic_note": note}


def kernel_sha1():
    # The persistent GEMM kernel's device code: the counters belong to it.
    with open(os.path.join(ROOT, "micro_polymerization_gb300", "csrc", "mp_kernel.cuh"), "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()


def roofline_us(g, peaks, d_bytes=4):
    t_flop = g.flops / (peaks["bf16_tflops"] * 1e6)
    t_mem = g.min_bytes(d_bytes) / (peaks["hbm_gbs"] * 1e3)
    return max(t_flop, t_mem), ("tensor" if t_flop >= t_mem else "hbm")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    _count = 0

    def __init__(self, index):
        self.index = index
        self.proc = None
        ClockSampler._count += 1
        self.path = os.path.join("/tmp", f"mp_clocks_{os.getpid()}_{ClockSampler._count}.csv")
        self._summary = None

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self._summary is None:
            self._summary = self._read()
        return self._summary

    def _read(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def rank_workload(name: str, rank: int):
    """Each rank runs its own copy of the workload (weak scaling): same shapes,
    operands seeded per rank.  ``shape:M,N,K[,beta]`` names a one-GEMM
    workload (alpha = 1, C uniform when beta != 0), for profiling one shape."""
    from micro_polymerization_gb300 import workloads as wl
    if name.startswith("shape:"):
        vals = [float(x) for x in name[len("shape:"):].split(",")]
        M, N, K = (int(v) for v in vals[:3])
        beta = vals[3] if len(vals) > 3 else 0.0
        gs = [wl.Gemm(M, N, K, alpha=1.0, beta=beta, seed=77)]
    elif name in wl.GROUPED_WORKLOADS:
        gs = wl.GROUPED_WORKLOADS[name]()
    else:
        gs = wl.workload(name)
    if rank == 0:
        return gs
    import dataclasses
    return [dataclasses.replace(g, seed=g.seed + 1_000_003 * rank) for g in gs]


def needs_repack(ptr: int, ld: int) -> bool:
    return ptr % 16 != 0 or (ld * 2) % 16 != 0


# ---------------------------------------------------------------------------
# call building and timing helpers
# ---------------------------------------------------------------------------
def gemm_call(lib, h, g, A, B, C, D, sp, epi=0):
    """Pre-marshalled C-ABI arguments of one GEMM (the call itself plans and
    launches)."""
    cp = C.data_ptr() if C is not None else None
    if g.batch > 1:
        return (lib.mp_gemm_batched, (h.ptr, g.batch, g.M, g.N, g.K, A.data_ptr(), g.K, g.M * g.K,
                                      B.data_ptr(), g.N, g.K * g.N, cp, g.N, g.M * g.N,
                                      D.data_ptr(), g.N, g.M * g.N, g.alpha, g.beta, sp))
    if epi:
        return (lib.mp_gemm_ex, (h.ptr, g.M, g.N, g.K, A.data_ptr(), g.K, B.data_ptr(), g.N,
                                 cp, g.N, D.data_ptr(), g.N, g.alpha, g.beta, epi, sp))
    return (lib.mp_gemm, (h.ptr, g.M, g.N, g.K, A.data_ptr(), g.K, B.data_ptr(), g.N,
                          cp, g.N, D.data_ptr(), g.N, g.alpha, g.beta, sp))


def new_output(g, dev, out_bf16=False):
    import torch
    return torch.empty((g.batch, g.M, g.N) if g.batch > 1 else (g.M, g.N), device=dev,
                       dtype=torch.bfloat16 if out_bf16 else torch.float32)


def run_calls(calls):
    import micro_polymerization_gb300 as mp
    for fn, a in calls:
        st = fn(*a)
        if st != 0:
            raise mp.MPError(st, "GEMM call")


def operand_bytes(ops_i):
    return sum(t.numel() * t.element_size() for t in ops_i if t is not None)


def per_shape_back_to_back(lib, h, gs, ops, sp, stream, epi=0, reps=3):
    """Device time per call of each GEMM when it is called back to back, as in
    a step, with cold operands: the calls cycle over copies of the GEMM's
    operands and outputs that together exceed twice L2 (at most 128 copies and
    about 4 GiB), so every call reads operands L2 no longer holds, except for
    GEMMs so small that 128 copies still fit.  The GPU is held by a sleep
    kernel while the calls are queued, so host issue time is not measured;
    events bracket the whole run of calls, not each call (an event between
    two calls costs about 5 us of device time here: it ends the programmatic
    overlap of one launch with the next).  Planning is inside every call (a
    plan-cache hit after the first)."""
    import torch
    out = []
    for g, o in zip(gs, ops):
        nbytes = operand_bytes(o)
        copies = int(min(128, max(2, math.ceil(2 * L2_BYTES / max(1, nbytes)))))
        copies = max(2, min(copies, int((4 << 30) // max(1, nbytes))))
        A, B, C, D = o
        sets = [o] + [(A.clone(), B.clone(), C.clone() if C is not None else None, torch.empty_like(D))
                      for _ in range(copies - 1)]
        calls = [gemm_call(lib, h, g, a, b, c, d, sp, epi) for a, b, c, d in sets]
        run_calls(calls)
        best = float("inf")
        for _ in range(reps):
            torch.cuda._sleep(20_000_000)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run_calls(calls)
            e1.record(stream)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) * 1e3 / len(calls))
        out.append(best)
        del sets, calls
    return np.array(out)


def flop_weighted_frac(gs, t_us, peaks, d_bytes=4):
    troof = np.array([roofline_us(g, peaks, d_bytes)[0] for g in gs])
    flops = np.array([g.flops for g in gs], dtype=np.float64)
    return float(np.sum(flops * troof / t_us) / np.sum(flops)), float(troof.sum() / t_us.sum())


CONFIG_RECORDS = ["single_skinny", "dynamic_resolution", "merged_qkv", "merged_batched", "stress"]


def config_record(name, args, lib, h, dev, sp, stream, peaks, local):
    """One line per further workload of the metric: the whole workload as one
    step of back-to-back calls (TFLOP/s, clocks sampled meanwhile) and the
    FLOP-weighted per-shape roofline fraction over at most 128 of its GEMMs
    (a seeded sample; the stress sweep keeps 4096^3)."""
    import torch
    from micro_polymerization_gb300 import workloads as wl
    gs = wl.workload(name)
    ops = []
    for g in gs:
        A, B, C = wl.make_operands(g, device=dev)
        ops.append((A, B, C, new_output(g, dev)))
    calls = [gemm_call(lib, h, g, *o, sp) for g, o in zip(gs, ops)]
    for _ in range(3):
        run_calls(calls)
    torch.cuda.synchronize()
    # Enough steps for the clock sampler (100 ms period) to see the region:
    # at least about 0.25 s, at least 3 steps.
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    run_calls(calls)
    w1.record(stream)
    torch.cuda.synchronize()
    est_ms = max(1e-3, w0.elapsed_time(w1))
    steps = int(max(3, min(20000, math.ceil(250.0 / est_ms))))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        e0.record(stream)
        for _ in range(steps):
            run_calls(calls)
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    flops = sum(g.flops for g in gs)
    idx = list(range(len(gs)))
    if len(gs) > 128:
        idx = sorted(np.random.default_rng(7).choice(len(gs) - 1, 127, replace=False).tolist()) + [len(gs) - 1]
    sub_g = [gs[i] for i in idx]
    t = per_shape_back_to_back(lib, h, sub_g, [ops[i] for i in idx], sp, stream)
    fw, ratio = flop_weighted_frac(sub_g, t, peaks)
    del ops, calls
    torch.cuda.empty_cache()
    return {"workload": workload_desc(name), "gemms": len(gs), "value": round(flops / (ms * 1e-3) / 1e12, 3),
            "unit": "TFLOPS", "ms_per_step": round(ms, 4), "steps": steps,
            "per_shape_roofline": {"flop_weighted_frac": round(fw, 4), "sum_troof_over_sum_t": round(ratio, 4),
                                   "gemms": len(sub_g)},
            "clocks": clocks.summary()}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def run_mp(args):
    import torch
    import micro_polymerization_gb300 as mp
    from micro_polymerization_gb300 import workloads as wl

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    # The planner's performance model: the table measured on GB300 by
    # micro_polymerization_gb300/calibrate.py and shipped with the package
    # (mp_init's default), or with --no-calib the analytic model.
    calib = calib_arg(args)
    h = mp.mp_init(local, calib)
    lib = mp.library()
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    gs = rank_workload(args.workload, rank)
    if args.limit:
        gs = gs[:args.limit]
    act, out_bf16 = EPILOGUES[args.epilogue]
    epi = act | (mp.MP_EPI_OUT_BF16 if out_bf16 else 0)
    d_bytes = 2 if out_bf16 else 4
    if epi and any(g.batch > 1 for g in gs):
        raise SystemExit("--epilogue applies to workloads of single GEMMs")
    ops = []
    launches_per_step = 0
    for g in gs:
        A, B, C = wl.make_operands(g, device=dev)
        D = torch.empty((g.batch, g.M, g.N) if g.batch > 1 else (g.M, g.N), device=dev,
                        dtype=torch.bfloat16 if out_bf16 else torch.float32)
        ops.append((g, A, B, C, D))
        launches_per_step += 1 + int(needs_repack(A.data_ptr(), g.K)) + int(needs_repack(B.data_ptr(), g.N))
    torch.cuda.synchronize()

    # Pre-marshalled C-ABI argument tuples (the call itself plans and launches).
    calls = [gemm_call(lib, h, g, A, B, C, D, sp, epi) for g, A, B, C, D in ops]

    def step(evs=None):
        for i, (fn, a) in enumerate(calls):
            if evs is not None:
                evs[i][0].record(stream)
            st = fn(*a)
            if st != 0:
                raise mp.MPError(st, "mp_gemm")
            if evs is not None:
                evs[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    if mp.mp_check(h) != 0:
        raise RuntimeError("device status word set during warm-up")
    torch.cuda.synchronize()

    # Per-launch device time of every GEMM (events around each call).
    n = len(calls)
    per_launch = np.zeros(n)
    reps = max(1, min(args.steps, 20))
    for _ in range(reps):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        step(evs)
        torch.cuda.synchronize()
        per_launch += np.array([a.elapsed_time(b) * 1e3 for a, b in evs])
    per_launch /= reps

    # The timed region: K whole steps, barrier + synchronize on both sides.
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    status = mp.mp_check(h)
    if status != 0:
        raise RuntimeError(f"device status word set in the timed region: {status}")
    elapsed_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    ms_per_step = elapsed_ms / args.steps
    flops_step = sum(g.flops for g in gs)
    value = flops_step * world * args.steps / (elapsed_ms * 1e-3) / 1e12

    # The same problems as one grouped submission (only when they are all
    # single GEMMs with the plain epilogue): informational, not the headline,
    # which times the separate calls above.
    as_group = None
    if not epi and all(g.batch == 1 for g in gs) and not args.no_group:
        arr = (mp.MpGemmProblem * len(ops))()
        for i, (g, A, B, C, D) in enumerate(ops):
            arr[i] = mp.MpGemmProblem(g.M, g.N, g.K, A.data_ptr(), g.K, B.data_ptr(), g.N,
                                      C.data_ptr() if C is not None else None, g.N, D.data_ptr(), g.N,
                                      g.alpha, g.beta)

        def group_step():
            st = lib.mp_gemm_grouped(h.ptr, len(ops), arr, sp)
            if st != 0:
                raise mp.MPError(st, "mp_gemm_grouped")

        for _ in range(3):
            group_step()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            group_step()
        g1.record(stream)
        torch.cuda.synchronize()
        ms_group = g0.elapsed_time(g1) / args.steps
        as_group = {"ms_per_step": round(ms_group, 4),
                    "value": round(sum(g.flops for g in gs) / (ms_group * 1e-3) / 1e12, 3),
                    "launches_per_step": -(-len(ops) // 48),
                    "note": "the same independent problems as one mp_gemm_grouped call per step; "
                            "not the headline, which times one mp_gemm call per problem"}
        if mp.mp_check(h) != 0:
            raise RuntimeError("device status word set by the grouped submission")

    # The same calls captured once in a CUDA graph and replayed: informational.
    # A replay runs the plans and operand addresses of the capture, so no
    # planning is inside it; the headline times the calls themselves.
    as_graph = None
    if not args.no_group:
        cs = torch.cuda.Stream(device=dev)
        gcalls = [gemm_call(lib, h, g, A, B, C, D, cs.cuda_stream, epi) for g, A, B, C, D in ops]
        with torch.cuda.stream(cs):
            run_calls(gcalls)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cs):
            run_calls(gcalls)
        with torch.cuda.stream(cs):
            for _ in range(3):
                graph.replay()
        torch.cuda.synchronize()
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(cs):
            r0.record(cs)
            for _ in range(args.steps):
                graph.replay()
            r1.record(cs)
        torch.cuda.synchronize()
        ms_graph = r0.elapsed_time(r1) / args.steps
        if mp.mp_check(h) != 0:
            raise RuntimeError("device status word set by the graph replays")
        as_graph = {"ms_per_step": round(ms_graph, 4),
                    "value": round(flops_step / (ms_graph * 1e-3) / 1e12, 3),
                    "note": "the same mp_gemm calls captured once in a CUDA graph and replayed; a replay "
                            "runs the plans and operand addresses of the capture (no planning inside); "
                            "not the headline"}
        del graph

    # Per-shape roofline fractions.  The per-shape time is the device time per
    # call with the GEMM called back to back on cold operands (see
    # per_shape_back_to_back); the event-bracketed times of the calls inside a
    # step (per_launch above) are reported beside it.
    b2b = per_shape_back_to_back(lib, h, gs, [o[1:] for o in ops], sp, stream, epi=epi)
    troof = np.array([roofline_us(g, peaks, d_bytes)[0] for g in gs])
    bounds = [roofline_us(g, peaks, d_bytes)[1] for g in gs]
    flops = np.array([g.flops for g in gs], dtype=np.float64)
    flop_weighted, time_ratio = flop_weighted_frac(gs, b2b, peaks, d_bytes)
    fw_events, ratio_events = flop_weighted_frac(gs, per_launch, peaks, d_bytes)

    # Dominant kernel: the persistent GEMM kernel (one launch per GEMM).  Its
    # bound is the one that dominates the summed roofline time.
    t_hbm = sum(t for t, b in zip(troof, bounds) if b == "hbm")
    t_ten = sum(t for t, b in zip(troof, bounds) if b == "tensor")
    if t_hbm >= t_ten:
        sel = [i for i, b in enumerate(bounds) if b == "hbm"]
        work = sum(gs[i].min_bytes(d_bytes) for i in sel)
        achieved = work / (b2b[sel].sum() * 1e-6) / 1e9
        peak = peaks["hbm_gbs"]
        unit, bound = "GB/s", "hbm"
    else:
        sel = [i for i, b in enumerate(bounds) if b == "tensor"]
        work = sum(gs[i].flops for i in sel)
        achieved = work / (b2b[sel].sum() * 1e-6) / 1e12
        peak = peaks["bf16_tflops"]
        unit, bound = "TFLOP/s", "tensor"
    traffic = traffic_fields(gs, sel, epi)

    # End to end: pinned host inputs copied in, outputs read back, every step.
    e2e = None
    if not args.no_e2e:
        host_in = []
        for g, A, B, C, D in ops:
            hA = torch.empty(A.shape, dtype=A.dtype, pin_memory=True); hA.copy_(A)
            hB = torch.empty(B.shape, dtype=B.dtype, pin_memory=True); hB.copy_(B)
            hC = None
            if C is not None:
                hC = torch.empty(C.shape, dtype=C.dtype, pin_memory=True); hC.copy_(C)
            hD = torch.empty(D.shape, dtype=D.dtype, pin_memory=True)
            host_in.append((hA, hB, hC, hD))
        h2d = sum(x.numel() * x.element_size() for t in host_in for x in t[:3] if x is not None)
        d2h = sum(t[3].numel() * t[3].element_size() for t in host_in)
        e2e_steps = max(1, min(args.steps, args.e2e_steps))

        # Three streams, as a serving loop would use them: host-to-device
        # copies, the GEMM calls (on the stream the calls were built for) and
        # device-to-host copies.  GEMM j waits only for its own inputs, and its
        # read-back only for GEMM j.  Across steps, a copy into an input waits
        # until the previous step's GEMM j has read it, and GEMM j waits until
        # the previous step's D_j has been read back.
        s_comp = stream
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        n_ops = len(ops)
        ev_in = [torch.cuda.Event() for _ in range(n_ops)]
        ev_done = [torch.cuda.Event() for _ in range(n_ops)]
        ev_back = [torch.cuda.Event() for _ in range(n_ops)]
        started = [False]

        def e2e_step():
            for j, ((g, A, B, C, D), (hA, hB, hC, hD), (fn, a)) in enumerate(zip(ops, host_in, calls)):
                with torch.cuda.stream(s_in):
                    if started[0]:
                        s_in.wait_event(ev_done[j])
                    A.copy_(hA, non_blocking=True)
                    B.copy_(hB, non_blocking=True)
                    if C is not None:
                        C.copy_(hC, non_blocking=True)
                    ev_in[j].record(s_in)
                s_comp.wait_event(ev_in[j])
                if started[0]:
                    s_comp.wait_event(ev_back[j])
                st = fn(*a)
                if st != 0:
                    raise mp.MPError(st, "mp_gemm")
                ev_done[j].record(s_comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_done[j])
                    hD.copy_(D, non_blocking=True)
                    ev_back[j].record(s_out)
            started[0] = True

        e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        torch.cuda.synchronize()
        t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
        e2e = {"value": round(flops_step * world * e2e_steps / t_e2e / 1e12, 3), "unit": "TFLOPS",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e2e_steps}

    # Planner latency: one mp_plan_many call over the workload's shapes on a
    # handle without a plan cache, so that every shape is searched; timed
    # around the single library call (no binding in the loop).
    plan_us = None
    if rank == 0:
        os.environ["MP_PLAN_CACHE"] = "0"
        try:
            h2 = mp.mp_init_host(mp.mp_get_hw(h)[0])
        finally:
            del os.environ["MP_PLAN_CACHE"]
        shapes = [(g.M, g.N, g.K) for g in gs if g.batch == 1]
        if shapes:
            mp.mp_plan_many(h2, shapes, want_plans=False)
            best = float("inf")
            for _ in range(20):
                t0 = time.perf_counter()
                mp.mp_plan_many(h2, shapes, want_plans=False)
                best = min(best, time.perf_counter() - t0)
            plan_us = best / len(shapes) * 1e6
        h2.close()

    # Informational: the same step on a handle without a plan cache, so that
    # every call runs the polymerizer's search before its launch.
    no_cache = None
    if not epi and rank == 0 and not args.no_group:
        os.environ["MP_PLAN_CACHE"] = "0"
        try:
            h3 = mp.mp_init(local, calib)
        finally:
            del os.environ["MP_PLAN_CACHE"]
        calls3 = [gemm_call(lib, h3, g, A, B, C, D, sp) for g, A, B, C, D in ops]
        for _ in range(3):
            run_calls(calls3)
        torch.cuda.synchronize()
        n0, n1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n0.record(stream)
        for _ in range(args.steps):
            run_calls(calls3)
        n1.record(stream)
        torch.cuda.synchronize()
        ms_nc = n0.elapsed_time(n1) / args.steps
        no_cache = {"ms_per_step": round(ms_nc, 4), "value": round(flops_step / (ms_nc * 1e-3) / 1e12, 3),
                    "note": "the same step on a handle made with MP_PLAN_CACHE=0: every call searches"}
        if mp.mp_check(h3) != 0:
            raise RuntimeError("device status word set by the no-cache step")
        h3.close()

    # The other workloads of the metric, one record each.
    configs = None
    if rank == 0 and args.workload == "dynamic_sequence" and not epi and not args.no_configs and not args.limit:
        configs = {name: config_record(name, args, lib, h, dev, sp, stream, peaks, local)
                   for name in CONFIG_RECORDS}

    if args.dump and rank == 0:
        with open(args.dump, "w") as f:
            for g, t, tr, b in zip(gs, per_launch, troof, bounds):
                p = mp.mp_plan_batched(h, g.batch, g.M, g.N, g.K)
                f.write(json.dumps({
                    "M": g.M, "N": g.N, "K": g.K, "batch": g.batch, "t_us": round(float(t), 3),
                    "troof_us": round(float(tr), 3), "frac": round(float(tr / t), 4), "bound": b,
                    "plan_cost_us": round(p.cost_us, 3), "regions": [
                        {"um": r.um, "un": r.un, "swap": r.swap, "m_ext": r.m_ext, "n_ext": r.n_ext,
                         "splits": r.splits, "tasks": r.f_parallel, "waves": r.f_wave}
                        for r in p.regions()]}) + "\n")

    cpu = cpu_baseline(args, gs, act=act, out_bf16=out_bf16) \
        if (rank == 0 and world == 1 and not args.no_cpu) else None
    if args.sweep and rank == 0:
        sweep(args, h, peaks, dev)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": run_config(args, gs, world),
            "per_shape_roofline": {"flop_weighted_frac": round(flop_weighted, 4),
                                   "sum_troof_over_sum_t": round(time_ratio, 4),
                                   "timing": "each GEMM called back to back on cold operands, events around "
                                             "the run of calls",
                                   "events_around_each_call": {"flop_weighted_frac": round(fw_events, 4),
                                                               "sum_troof_over_sum_t": round(ratio_events, 4)},
                                   "peaks": peak_src},
            "roofline": dict({"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                              "frac": round(achieved / peak, 4)}, **traffic,
                             launches=len(sel), kernel="k_poly_gemm", peak_source=peak_src),
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
            "as_one_group": as_group,
            "as_graph": as_graph,
            "plan_us": round(plan_us, 3) if plan_us is not None else None,
            "plan_how": "one mp_plan_many call over the workload's shapes, no plan cache, best of 20",
            "no_plan_cache": no_cache,
            "configs": configs,
            "cost_model": "calibrated" if calib else "analytic",
            "cost_model_table": os.path.relpath(calib, ROOT) if calib else None,
            "clocks": clocks.summary(), "impl": "mp",
        }
        print(json.dumps(line), flush=True)
    h.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


L2_BYTES = 126 * 2 ** 20


def run_config(args, gs, world):
    """The `config` object of the JSON line (the same for both arms)."""
    return {"workload": workload_desc(args.workload), "gemms_per_step": len(gs),
            "flops_per_step": int(sum(g.flops for g in gs)), "l2": l2_note(gs), "epilogue": args.epilogue,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def l2_note(gs):
    """How the timed region treats L2: the default workload touches far more
    distinct operand bytes per step than L2 holds; a one-shape workload does
    not, so its numbers are warm-L2 numbers (used for profiling only)."""
    total = sum(g.min_bytes() for g in gs)
    if total >= 2 * L2_BYTES:
        return f"inputs larger than L2 ({total / 1e9:.2f} GB of distinct operands per step)"
    return f"inputs smaller than L2 ({total / 1e9:.3f} GB per step, not flushed): warm-L2 numbers"


def workload_desc(name):
    if name.startswith("b2bshape:"):
        return f"one fused back-to-back GEMM (M,N0,N1,K0[,act0]) = ({name[len('b2bshape:'):]})"
    if name.startswith("shape:"):
        return f"single GEMM (M,N,K[,beta]) = ({name[len('shape:'):]}), alpha=1"
    return {
        "dynamic_sequence": "dynamic sequence length: 64 GEMMs, M = 8*seq (seq uniform [1,512]), "
                            "(N,K) cycling (2304,768),(768,768),(3072,768),(768,3072), bf16 A,B, beta=0",
        "single_skinny": "single GEMM (105,1024,12544), alpha=1, beta=1",
        "dynamic_resolution": "conv-as-GEMM, 64 draws of ResNet-50-like 3x3 layers",
        "merged_qkv": "A x concat(Wq,Wk,Wv), K=1024, N=3072, M uniform [1,4096], 64 draws",
        "merged_batched": "batched 12 x (seq,seq,64), seq uniform [16,512], 64 draws",
        "stress": "1000 log-uniform shapes in [1,16384]^3 plus 4096^3, alpha=1.5, beta=0.5",
        "grouped_experts": "grouped GEMM: 48 expert problems of one layer, M uniform [1,512], (N,K) = (2048,1024), "
                           "one mp_gemm_grouped call",
        "conv_resolution": "implicit-GEMM convolutions, the 64 dynamic-resolution layers as 3x3 stride-1 "
                           "NHWC convolutions",
        "b2b_adapter": "fused back-to-back GEMMs, 64 problems, M = 8*seq (seq uniform [1,512]), "
                       "768 -> 256 (ReLU) -> 768, bf16 A0,W0,W1, beta0=beta1=0",
        "b2b_1x1": "fused back-to-back GEMMs as two 1x1 convolutions, 64 problems, M = batch*H*W "
                   "(batch [1,32], H=W in {7,14,28,56}), 256 -> 64 (ReLU) -> 256",
    }[name]


def sweep(args, h, peaks, dev):
    """One summary line per workload on stderr (per-shape events, L2 flushed)."""
    import torch
    import micro_polymerization_gb300 as mp
    from micro_polymerization_gb300 import workloads as wl
    flush = torch.empty(int(512 * 2 ** 20), dtype=torch.uint8, device=dev)
    for name in wl.WORKLOADS:
        gs = wl.workload(name)
        if len(gs) > args.sweep_count:
            # A seeded sample of the list (the stress sweep's 4096^3 is kept).
            idx = np.random.default_rng(7).choice(len(gs) - 1, args.sweep_count - 1, replace=False)
            gs = [gs[i] for i in sorted(idx)] + [gs[-1]]
        ts, trs, fl = [], [], []
        for g in gs:
            A, B, C = wl.make_operands(g, device=dev)
            D = torch.empty((g.batch, g.M, g.N) if g.batch > 1 else (g.M, g.N), device=dev)
            fn = (lambda: mp.mp_gemm_batched(h, A, B, C, D, g.alpha, g.beta)) if g.batch > 1 else \
                 (lambda: mp.mp_gemm(h, A, B, C, D, g.alpha, g.beta))
            for _ in range(3):
                fn()
            best = []
            for _ in range(5):
                flush.random_(0, 255)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                best.append(e0.elapsed_time(e1) * 1e3)
            t = statistics.median(best)
            ts.append(t); trs.append(roofline_us(g, peaks)[0]); fl.append(g.flops)
            del A, B, C, D
        ts, trs, fl = map(np.array, (ts, trs, fl))
        frac = trs / ts
        sys.stderr.write(json.dumps({
            "workload": name, "gemms": len(gs), "tflops": round(fl.sum() / (ts.sum() * 1e-6) / 1e12, 2),
            "flop_weighted_roofline_frac": round(float((fl * frac).sum() / fl.sum()), 4),
            "sum_troof_over_sum_t": round(float(trs.sum() / ts.sum()), 4),
            "median_frac": round(float(np.median(frac)), 4), "min_frac": round(float(frac.min()), 4),
        }) + "\n")
        sys.stderr.flush()


# ---------------------------------------------------------------------------
# the CPU oracle, timed on a bounded sample of the same workload
# ---------------------------------------------------------------------------
def cpu_baseline(args, gs, budget_s=None, act=0, out_bf16=False):
    import torch
    import oracle
    from micro_polymerization_gb300 import workloads as wl
    budget_s = budget_s or args.cpu_seconds
    flops = 0.0
    used = 0
    t_total = 0.0
    done = 0
    for g in gs:
        A, B, C = wl.make_operands(g)
        if g.batch > 1:
            A, B = A[0], B[0]
            C = C[0] if C is not None else None
        rows = min(g.M, 256)
        Ab = wl.bf16_bits(A[:rows])
        Bb = wl.bf16_bits(B)
        Cn = C[:rows].numpy() if C is not None else None
        t0 = time.perf_counter()
        Dr, used = oracle.gemm_rows(Ab, Bb, Cn, g.alpha, g.beta)
        if act:
            Dr = oracle.epilogue(Dr, act)
        if out_bf16:
            Dr = oracle.bf16_round(Dr)
        t_total += time.perf_counter() - t0
        flops += 2.0 * rows * g.N * g.K
        done += 1
        if t_total >= budget_s:
            break
    return {"value": round(flops / t_total / 1e12, 6), "unit": "TFLOPS", "cores": int(used), "kind": "oracle",
            "seconds": round(t_total, 4),
            "sample": f"first min(M, 256) rows of each of the first {done} GEMMs of the workload "
                      f"({flops / 1e9:.1f} GFLOP in {t_total:.1f} s, fp64, OpenMP)"}


def grouped_names():
    from micro_polymerization_gb300 import workloads as wl
    return set(wl.GROUPED_WORKLOADS)


def is_conv(name: str) -> bool:
    from micro_polymerization_gb300 import workloads as wl
    return name in wl.CONV_WORKLOADS or name.startswith("convshape:")


def conv_workload(name: str):
    """A named convolution workload, or ``convshape:N,H,W,C,K`` for one 3x3
    'same' layer (alpha = 1, beta = 0), for profiling one shape."""
    from micro_polymerization_gb300 import workloads as wl
    if name.startswith("convshape:"):
        v = [int(x) for x in name[len("convshape:"):].split(",")]
        return [wl.Conv(v[0], v[1], v[2], v[3], v[4], seed=79)]
    return wl.CONV_WORKLOADS[name]()


def is_b2b(name: str) -> bool:
    from micro_polymerization_gb300 import workloads as wl
    return name in wl.B2B_WORKLOADS or name.startswith("b2bshape:")


def b2b_workload(name: str):
    """A named fused-pair workload, or ``b2bshape:M,N0,N1,K0[,act0]`` for one
    problem (alpha = 1, beta = 0), for profiling one shape."""
    from micro_polymerization_gb300 import workloads as wl
    if name.startswith("b2bshape:"):
        v = [int(x) for x in name[len("b2bshape:"):].split(",")]
        return [wl.B2B(v[0], v[1], v[2], v[3], act0=v[4] if len(v) > 4 else 0, seed=78)]
    return wl.B2B_WORKLOADS[name]()


def cpu_baseline_b2b(args, bs, budget_s=None):
    """The oracle's fused-pair evaluation on the first min(M, 256) rows of each
    problem (first GEMM in C over OpenMP rows, second a numpy fp64 product)."""
    import oracle
    from micro_polymerization_gb300 import workloads as wl
    budget_s = budget_s or args.cpu_seconds
    flops = t_total = 0.0
    done = 0
    for b in bs:
        A0, W0, C0, W1, C1 = wl.make_b2b_operands(b)
        rows = min(b.M, 256)
        a0, w0, w1 = wl.bf16_bits(A0[:rows]), wl.bf16_bits(W0), wl.bf16_bits(W1)
        c0 = C0[:rows].numpy() if C0 is not None else None
        c1 = C1[:rows].numpy() if C1 is not None else None
        t0 = time.perf_counter()
        oracle.b2b(a0, w0, c0, w1, c1, b.alpha0, b.beta0, b.alpha1, b.beta1, b.act0)
        t_total += time.perf_counter() - t0
        flops += 2.0 * rows * (b.N0 * b.K0 + b.N1 * b.N0)
        done += 1
        if t_total >= budget_s:
            break
    return {"value": round(flops / t_total / 1e12, 6), "unit": "TFLOPS", "seconds": round(t_total, 4), "cores": int(oracle.max_threads()),
            "kind": "oracle",
            "sample": f"first min(M, 256) rows of each of the first {done} problems of the workload "
                      f"({flops / 1e9:.1f} GFLOP in {t_total:.1f} s, fp64)"}


def run_b2b(args):
    """Fused back-to-back GEMMs (mp_gemm_b2b), one call per problem, back to
    back on one stream; the unfused pair (mp_gemm_ex writing a bf16 D0 with
    the activation, then mp_gemm) is timed beside it on the same operands."""
    import torch
    import micro_polymerization_gb300 as mp
    from micro_polymerization_gb300 import workloads as wl

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    h = mp.mp_init(local)
    lib = mp.library()
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    bs = b2b_workload(args.workload)
    if rank > 0:
        import dataclasses
        bs = [dataclasses.replace(b, seed=b.seed + 1_000_003 * rank) for b in bs]
    ops = []
    for b in bs:
        t = [x.to(dev) if x is not None else None for x in wl.make_b2b_operands(b)]
        D1 = torch.empty(b.M, b.N1, device=dev)
        D0 = torch.empty(b.M, b.N0, device=dev, dtype=torch.bfloat16)
        ops.append((b, *t, D1, D0))
    torch.cuda.synchronize()
    ptr = lambda x: x.data_ptr() if x is not None else None
    fused, unfused = [], []
    for b, A0, W0, C0, W1, C1, D1, D0 in ops:
        fused.append((lib.mp_gemm_b2b, (h.ptr, b.M, b.N0, b.N1, b.K0, A0.data_ptr(), b.K0, W0.data_ptr(), b.N0,
                                        ptr(C0), b.N0, W1.data_ptr(), b.N1, ptr(C1), b.N1, D1.data_ptr(), b.N1,
                                        b.alpha0, b.beta0, b.alpha1, b.beta1, b.act0, sp)))
        unfused.append((lib.mp_gemm_ex, (h.ptr, b.M, b.N0, b.K0, A0.data_ptr(), b.K0, W0.data_ptr(), b.N0, ptr(C0),
                                         b.N0, D0.data_ptr(), b.N0, b.alpha0, b.beta0,
                                         b.act0 | mp.MP_EPI_OUT_BF16, sp)))
        unfused.append((lib.mp_gemm, (h.ptr, b.M, b.N1, b.N0, D0.data_ptr(), b.N0, W1.data_ptr(), b.N1, ptr(C1),
                                      b.N1, D1.data_ptr(), b.N1, b.alpha1, b.beta1, sp)))

    def step(calls, evs=None):
        for i, (fn, a) in enumerate(calls):
            if evs is not None:
                evs[i][0].record(stream)
            st = fn(*a)
            if st != 0:
                raise mp.MPError(st, fn.__name__)
            if evs is not None:
                evs[i][1].record(stream)

    def timed(calls, steps):
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step(calls)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(e0.elapsed_time(e1), world, dev) / steps

    for _ in range(args.warmup):
        step(fused)
        step(unfused)
    torch.cuda.synchronize()
    if mp.mp_check(h) != 0:
        raise RuntimeError("device status word set during warm-up")
    # The fused kernel itself (forced), per launch, for its roofline.
    mp.mp_set_b2b_mode(h, mp.MP_B2B_FUSED)
    step(fused)
    n = len(fused)
    per_launch = np.zeros(n)
    reps = max(1, min(args.steps, 20))
    for _ in range(reps):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        step(fused, evs)
        torch.cuda.synchronize()
        per_launch += np.array([a.elapsed_time(b) * 1e3 for a, b in evs])
    per_launch /= reps
    ms_kernel = timed(fused, args.steps)
    mp.mp_set_b2b_mode(h, mp.MP_B2B_AUTO)
    modes = [mp.mp_plan_b2b(h, b.M, b.N0, b.N1, b.K0).mode for b in bs]
    step(fused)
    with ClockSampler(local) as clocks:
        ms_step = timed(fused, args.steps)
    ms_unfused = timed(unfused, args.steps)
    if mp.mp_check(h) != 0:
        raise RuntimeError("device status word set in the timed region")
    flops_step = sum(b.flops for b in bs)
    value = flops_step * world / (ms_step * 1e-3) / 1e12

    t_flop = np.array([b.flops / (peaks["bf16_tflops"] * 1e6) for b in bs])
    t_mem = np.array([b.min_bytes() / (peaks["hbm_gbs"] * 1e3) for b in bs])
    troof = np.maximum(t_flop, t_mem)
    if t_flop.sum() >= t_mem.sum():
        bound, unit, peak = "tensor", "TFLOP/s", peaks["bf16_tflops"]
        achieved = flops_step / (per_launch.sum() * 1e-6) / 1e12
    else:
        bound, unit, peak = "hbm", "GB/s", peaks["hbm_gbs"]
        achieved = sum(b.min_bytes() for b in bs) / (per_launch.sum() * 1e-6) / 1e9
    flops = np.array([b.flops for b in bs], dtype=np.float64)
    flop_weighted = float(np.sum(flops * troof / per_launch) / np.sum(flops))

    e2e = None
    if not args.no_e2e:
        host = []
        for b, A0, W0, C0, W1, C1, D1, D0 in ops:
            hx = []
            for x in (A0, W0, C0, W1, C1, D1):
                if x is None:
                    hx.append(None)
                    continue
                y = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
                y.copy_(x)
                hx.append(y)
            host.append(hx)
        h2d = sum(x.numel() * x.element_size() for hx in host for x in hx[:5] if x is not None)
        d2h = sum(hx[5].numel() * hx[5].element_size() for hx in host)

        def e2e_step():
            for (b, A0, W0, C0, W1, C1, D1, D0), hx, (fn, a) in zip(ops, host, fused):
                for dst, src in zip((A0, W0, C0, W1, C1), hx[:5]):
                    if dst is not None:
                        dst.copy_(src, non_blocking=True)
                st = fn(*a)
                if st != 0:
                    raise mp.MPError(st, "mp_gemm_b2b")
                hx[5].copy_(D1, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        e2e_steps = max(1, min(args.steps, args.e2e_steps))
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        torch.cuda.synchronize()
        t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
        e2e = {"value": round(flops_step * world * e2e_steps / t_e2e / 1e12, 3), "unit": "TFLOPS",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e2e_steps}

    cpu = cpu_baseline_b2b(args, bs) if (rank == 0 and world == 1 and not args.no_cpu) else None
    if rank == 0:
        b0 = bs[0]
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": workload_desc(args.workload), "problems_per_step": len(bs),
                       "shape": {"N0": b0.N0, "N1": b0.N1, "K0": b0.K0, "act0": b0.act0},
                       "flops_per_step": int(flops_step),
                       "l2": "inputs larger than L2" if sum(b.min_bytes() for b in bs) > L2_BYTES else
                             "inputs smaller than L2",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "unfused": {"ms_per_step": round(ms_unfused, 4),
                        "value": round(flops_step * world / (ms_unfused * 1e-3) / 1e12, 3),
                        "calls": "mp_gemm_ex (bf16 D0, activation) + mp_gemm",
                        "fused_speedup": round(ms_unfused / ms_step, 3)},
            "forms": {"fused_kernel": modes.count(mp.MP_B2B_FUSED),
                      "two_launch": modes.count(mp.MP_B2B_TWO_LAUNCH),
                      "fused_kernel_only_ms_per_step": round(ms_kernel, 4),
                      "note": "value times mp_gemm_b2b with its automatic choice of form per problem"},
            "per_shape_roofline": {"flop_weighted_frac": round(flop_weighted, 4),
                                   "sum_troof_over_sum_t": round(float(troof.sum() / per_launch.sum()), 4),
                                   "peaks": peak_src},
            "roofline": {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                         "frac": round(achieved / peak, 4), "traffic": None, "launches": n,
                         "kernel": "k_b2b_gemm", "peak_source": peak_src},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": n * args.steps,
            "clocks": clocks.summary(), "impl": "mp",
        }
        print(json.dumps(line), flush=True)
    h.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def cpu_baseline_conv(args, cs, budget_s=None):
    """The oracle's convolution on the first image of each layer."""
    import oracle
    from micro_polymerization_gb300 import workloads as wl
    budget_s = budget_s or args.cpu_seconds
    flops = t_total = 0.0
    done = 0
    for c in cs:
        X, F, Cin = wl.make_conv_operands(c)
        xb, fb = wl.bf16_bits(X[:1]), wl.bf16_bits(F)
        cn = Cin[:1].numpy() if Cin is not None else None
        t0 = time.perf_counter()
        oracle.conv2d_nhwc(xb, fb, cn, c.alpha, c.beta, c.pad_h, c.pad_w)
        t_total += time.perf_counter() - t0
        flops += c.flops / c.N
        done += 1
        if t_total >= budget_s:
            break
    import os as _os
    return {"value": round(flops / t_total / 1e12, 6), "unit": "TFLOPS", "seconds": round(t_total, 4), "cores": int(_os.cpu_count() or 1),
            "kind": "oracle",
            "sample": f"first image of each of the first {done} layers ({flops / 1e9:.1f} GFLOP in "
                      f"{t_total:.1f} s, fp64, numpy products per filter tap)"}


def run_conv(args):
    """Implicit-GEMM convolutions (mp_conv2d), one call per layer, back to back
    on one stream; mp_gemm on each layer's prebuilt im2col matrix (the GEMM a
    GEMM-based convolution runs) is timed beside it."""
    import torch
    import torch.nn.functional as tnf
    import micro_polymerization_gb300 as mp
    from micro_polymerization_gb300 import workloads as wl

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    h = mp.mp_init(local, calib_arg(args))
    lib = mp.library()
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    cs = conv_workload(args.workload)
    if rank > 0:
        import dataclasses
        cs = [dataclasses.replace(c, seed=c.seed + 1_000_003 * rank) for c in cs]
    ops, conv_calls, gemm_calls = [], [], []
    for c in cs:
        X, F, Cin = [t.to(dev) if t is not None else None for t in wl.make_conv_operands(c)]
        D = torch.empty(c.N, c.P, c.Q, c.K, device=dev)
        # The GEMM path's operands: im2col in (c, r, s) column order (unfold's),
        # the filter permuted to match.
        A = tnf.unfold(X.permute(0, 3, 1, 2).float(), (c.R, c.S), padding=(c.pad_h, c.pad_w))
        A = A.transpose(1, 2).reshape(c.N * c.P * c.Q, c.C * c.R * c.S).to(torch.bfloat16).contiguous()
        B = F.permute(2, 0, 1, 3).reshape(c.C * c.R * c.S, c.K).contiguous()
        Dg = torch.empty(c.N * c.P * c.Q, c.K, device=dev)
        ops.append((c, X, F, Cin, D, A, B, Dg))
        conv_calls.append((lib.mp_conv2d, (h.ptr, c.N, c.H, c.W, c.C, c.K, c.R, c.S, c.pad_h, c.pad_w,
                                           X.data_ptr(), F.data_ptr(), Cin.data_ptr() if Cin is not None else None,
                                           c.K, D.data_ptr(), c.K, c.alpha, c.beta, sp)))
        gemm_calls.append((lib.mp_gemm, (h.ptr, A.shape[0], c.K, A.shape[1], A.data_ptr(), A.shape[1],
                                         B.data_ptr(), c.K, None, c.K, Dg.data_ptr(), c.K, c.alpha, 0.0, sp)))
    torch.cuda.synchronize()

    def step(calls, evs=None):
        for i, (fn, a) in enumerate(calls):
            if evs is not None:
                evs[i][0].record(stream)
            st = fn(*a)
            if st != 0:
                raise mp.MPError(st, fn.__name__)
            if evs is not None:
                evs[i][1].record(stream)

    def timed(calls, steps):
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step(calls)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(e0.elapsed_time(e1), world, dev) / steps

    for _ in range(args.warmup):
        step(conv_calls)
        step(gemm_calls)
    torch.cuda.synchronize()
    if mp.mp_check(h) != 0:
        raise RuntimeError("device status word set during warm-up")
    n = len(conv_calls)
    per_launch = np.zeros(n)
    reps = max(1, min(args.steps, 20))
    for _ in range(reps):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        step(conv_calls, evs)
        torch.cuda.synchronize()
        per_launch += np.array([a.elapsed_time(b) * 1e3 for a, b in evs])
    per_launch /= reps
    with ClockSampler(local) as clocks:
        ms_step = timed(conv_calls, args.steps)
    ms_gemm = timed(gemm_calls, args.steps)
    if args.dump and rank == 0:
        per_gemm = np.zeros(n)
        for _ in range(reps):
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
            step(gemm_calls, evs)
            torch.cuda.synchronize()
            per_gemm += np.array([a.elapsed_time(b) * 1e3 for a, b in evs])
        per_gemm /= reps
        with open(args.dump, "w") as f:
            for c, t, tg in zip(cs, per_launch, per_gemm):
                pl = mp.mp_plan_conv(h, c.N, c.H, c.W, c.C, c.K, c.R, c.S, c.pad_h, c.pad_w)
                f.write(json.dumps({"N": c.N, "H": c.H, "C": c.C, "K": c.K, "t_us": round(float(t), 2),
                                    "gemm_us": round(float(tg), 2), "wb": pl.wb, "hb": pl.hb, "nb": pl.nb,
                                    "bn": pl.bn, "units": pl.units, "ksteps": pl.ksteps,
                                    "useful": round(pl.useful, 3), "model_us": round(pl.cost_us, 2)}) + "\n")
    if mp.mp_check(h) != 0:
        raise RuntimeError("device status word set in the timed region")
    flops_step = sum(c.flops for c in cs)
    value = flops_step * world / (ms_step * 1e-3) / 1e12
    t_flop = np.array([c.flops / (peaks["bf16_tflops"] * 1e6) for c in cs])
    t_mem = np.array([c.min_bytes() / (peaks["hbm_gbs"] * 1e3) for c in cs])
    troof = np.maximum(t_flop, t_mem)
    if t_flop.sum() >= t_mem.sum():
        bound, unit, peak = "tensor", "TFLOP/s", peaks["bf16_tflops"]
        achieved = flops_step / (per_launch.sum() * 1e-6) / 1e12
    else:
        bound, unit, peak = "hbm", "GB/s", peaks["hbm_gbs"]
        achieved = sum(c.min_bytes() for c in cs) / (per_launch.sum() * 1e-6) / 1e9
    flops = np.array([c.flops for c in cs], dtype=np.float64)
    flop_weighted = float(np.sum(flops * troof / per_launch) / np.sum(flops))

    e2e = None
    if not args.no_e2e:
        host = []
        for (c, X, F, Cin, D, A, B, Dg) in ops:
            hx = []
            for x in (X, F, Cin, D):
                if x is None:
                    hx.append(None)
                    continue
                y = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
                y.copy_(x)
                hx.append(y)
            host.append(hx)
        h2d = sum(x.numel() * x.element_size() for hx in host for x in hx[:3] if x is not None)
        d2h = sum(hx[3].numel() * hx[3].element_size() for hx in host)

        def e2e_step():
            for (c, X, F, Cin, D, A, B, Dg), hx, (fn, a) in zip(ops, host, conv_calls):
                for dst, src in zip((X, F, Cin), hx[:3]):
                    if dst is not None:
                        dst.copy_(src, non_blocking=True)
                st = fn(*a)
                if st != 0:
                    raise mp.MPError(st, "mp_conv2d")
                hx[3].copy_(D, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        e2e_steps = max(1, min(args.steps, args.e2e_steps))
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        torch.cuda.synchronize()
        t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
        e2e = {"value": round(flops_step * world * e2e_steps / t_e2e / 1e12, 3), "unit": "TFLOPS",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e2e_steps}

    cpu = cpu_baseline_conv(args, cs) if (rank == 0 and world == 1 and not args.no_cpu) else None
    if rank == 0:
        im2col_bytes = sum(2 * c.N * c.P * c.Q * c.R * c.S * c.C for c in cs)
        x_bytes = sum(2 * c.N * c.H * c.W * c.C for c in cs)
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "implicit-GEMM convolutions of the dynamic-resolution workload: 64 3x3 "
                                   "stride-1 'same' layers, NHWC, batch [1,32], C = K = 64*2^s",
                       "layers_per_step": len(cs), "flops_per_step": int(flops_step),
                       "l2": "inputs larger than L2" if sum(c.min_bytes() for c in cs) > L2_BYTES else
                             "inputs smaller than L2",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "gemm_on_im2col": {"ms_per_step": round(ms_gemm, 4),
                               "value": round(flops_step * world / (ms_gemm * 1e-3) / 1e12, 3),
                               "calls": "mp_gemm on each layer's prebuilt im2col matrix (building it not timed)",
                               "im2col_bytes_per_step": int(im2col_bytes), "x_bytes_per_step": int(x_bytes),
                               "implicit_speedup": round(ms_gemm / ms_step, 3)},
            "per_shape_roofline": {"flop_weighted_frac": round(flop_weighted, 4),
                                   "sum_troof_over_sum_t": round(float(troof.sum() / per_launch.sum()), 4),
                                   "peaks": peak_src},
            "roofline": {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                         "frac": round(achieved / peak, 4), "traffic": None, "launches": n,
                         "kernel": "k_conv_igemm", "peak_source": peak_src},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": n * args.steps,
            "clocks": clocks.summary(), "impl": "mp",
        }
        print(json.dumps(line), flush=True)
    h.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_grouped(args):
    """A group of problems of different shapes as one mp_gemm_grouped call per
    step; the same problems as separate mp_gemm calls are timed beside it."""
    import ctypes
    import torch
    import micro_polymerization_gb300 as mp
    from micro_polymerization_gb300 import workloads as wl

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    h = mp.mp_init(local, calib_arg(args))
    lib = mp.library()
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    gs = rank_workload(args.workload, rank)
    ops = []
    for g in gs:
        A, B, C = wl.make_operands(g, device=dev)
        ops.append((g, A, B, C, torch.empty(g.M, g.N, device=dev)))
    torch.cuda.synchronize()
    arr = (mp.MpGemmProblem * len(ops))()
    singles = []
    for i, (g, A, B, C, D) in enumerate(ops):
        cp = C.data_ptr() if C is not None else None
        arr[i] = mp.MpGemmProblem(g.M, g.N, g.K, A.data_ptr(), g.K, B.data_ptr(), g.N, cp, g.N, D.data_ptr(), g.N,
                                  g.alpha, g.beta)
        singles.append((h.ptr, g.M, g.N, g.K, A.data_ptr(), g.K, B.data_ptr(), g.N, cp, g.N, D.data_ptr(), g.N,
                        g.alpha, g.beta, sp))
    count = len(ops)

    def grouped_step():
        st = lib.mp_gemm_grouped(h.ptr, count, arr, sp)
        if st != 0:
            raise mp.MPError(st, "mp_gemm_grouped")

    def singles_step():
        for a in singles:
            st = lib.mp_gemm(*a)
            if st != 0:
                raise mp.MPError(st, "mp_gemm")

    def timed(fn, steps):
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(e0.elapsed_time(e1), world, dev) / steps

    for _ in range(args.warmup):
        grouped_step()
        singles_step()
    torch.cuda.synchronize()
    if mp.mp_check(h) != 0:
        raise RuntimeError("device status word set during warm-up")
    with ClockSampler(local) as clocks:
        ms_step = timed(grouped_step, args.steps)
    ms_single = timed(singles_step, args.steps)
    if mp.mp_check(h) != 0:
        raise RuntimeError("device status word set in the timed region")
    flops_step = sum(g.flops for g in gs)
    bytes_step = sum(g.min_bytes() for g in gs)
    value = flops_step * world / (ms_step * 1e-3) / 1e12
    t_flop = flops_step / (peaks["bf16_tflops"] * 1e6)
    t_mem = bytes_step / (peaks["hbm_gbs"] * 1e3)
    launches = -(-count // 48)
    if t_flop >= t_mem:
        bound, unit, peak, achieved = "tensor", "TFLOP/s", peaks["bf16_tflops"], flops_step / (ms_step * 1e-3) / 1e12
    else:
        bound, unit, peak, achieved = "hbm", "GB/s", peaks["hbm_gbs"], bytes_step / (ms_step * 1e-3) / 1e9
    e2e = None
    if not args.no_e2e:
        host = []
        for (g, A, B, C, D) in ops:
            hx = []
            for x in (A, B, C, D):
                if x is None:
                    hx.append(None)
                    continue
                y = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
                y.copy_(x)
                hx.append(y)
            host.append(hx)
        h2d = sum(x.numel() * x.element_size() for hx in host for x in hx[:3] if x is not None)
        d2h = sum(hx[3].numel() * hx[3].element_size() for hx in host)

        def e2e_step():
            for (g, A, B, C, D), hx in zip(ops, host):
                for dst, src in zip((A, B, C), hx[:3]):
                    if dst is not None:
                        dst.copy_(src, non_blocking=True)
            grouped_step()
            for (g, A, B, C, D), hx in zip(ops, host):
                hx[3].copy_(D, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        e2e_steps = max(1, min(args.steps, args.e2e_steps))
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        torch.cuda.synchronize()
        t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
        e2e = {"value": round(flops_step * world * e2e_steps / t_e2e / 1e12, 3), "unit": "TFLOPS",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e2e_steps}
    cpu = cpu_baseline(args, gs) if (rank == 0 and world == 1 and not args.no_cpu) else None
    if rank == 0:
        plan = mp.mp_plan_grouped(h, [(g.M, g.N, g.K) for g in gs])
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": workload_desc(args.workload), "problems_per_step": count,
                       "flops_per_step": int(flops_step), "bn": plan.bn, "launches_per_step": launches,
                       "l2": "inputs larger than L2" if bytes_step > L2_BYTES else "inputs smaller than L2",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "separate_calls": {"ms_per_step": round(ms_single, 4),
                               "value": round(flops_step * world / (ms_single * 1e-3) / 1e12, 3),
                               "calls": f"{count} mp_gemm calls", "grouped_speedup": round(ms_single / ms_step, 3)},
            "roofline": {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                         "frac": round(achieved / peak, 4), "traffic": None, "launches": launches,
                         "kernel": "k_gemm_grouped", "peak_source": peak_src},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches * args.steps,
            "clocks": clocks.summary(), "impl": "mp",
        }
        print(json.dumps(line), flush=True)
    h.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from micro_polymerization_gb300 import workloads as wl
    import oracle  # noqa: F401
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps))
    config = {"workload": workload_desc(args.workload), "epilogue": args.epilogue}
    if is_conv(args.workload):
        cs = conv_workload(args.workload)
        for _ in range(args.warmup):
            cpu_baseline_conv(args, cs[:1], budget_s=0.01)
        vals = [cpu_baseline_conv(args, cs, budget_s=per_step) for _ in range(args.steps)]
    elif is_b2b(args.workload):
        bs = b2b_workload(args.workload)
        for _ in range(args.warmup):
            cpu_baseline_b2b(args, bs[:1], budget_s=0.01)
        vals = [cpu_baseline_b2b(args, bs, budget_s=per_step) for _ in range(args.steps)]
    else:
        gs = rank_workload(args.workload, 0)
        for _ in range(args.warmup):
            cpu_baseline(args, gs[:1], budget_s=0.01)
        act, out_bf16 = EPILOGUES[args.epilogue]
        vals = [cpu_baseline(args, gs, budget_s=per_step, act=act, out_bf16=out_bf16) for _ in range(args.steps)]
        config = run_config(args, gs, world)
    v = statistics.median(x["value"] for x in vals)
    # A step of this arm is a bounded sample of the workload: its time is the
    # sample's wall time.
    ms_step = statistics.median(x["seconds"] for x in vals) * 1e3
    line = {
        "metric": METRIC, "value": v, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": v, "unit": "TFLOPS", "cores": vals[0]["cores"], "kind": "oracle",
                         "sample": vals[0]["sample"]},
        "e2e": {"value": v, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "impl": "reference",
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["mp", "reference"], default="mp")
    ap.add_argument("--workload", default="dynamic_sequence")
    ap.add_argument("--epilogue", choices=sorted(EPILOGUES), default="none",
                    help="activation and D type of every GEMM (mp_gemm_ex); none = mp_gemm")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--sweep-count", type=int, default=128, help="GEMMs per workload in the sweep (sampled)")
    ap.add_argument("--dump", default=None, help="write per-GEMM time, roofline and plan (JSON lines)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-group", action="store_true",
                    help="skip the informational grouped submission and CUDA-graph replay")
    ap.add_argument("--no-calib", action="store_true", help="plan with the analytic cost model")
    ap.add_argument("--no-configs", action="store_true", help="skip the records of the other workloads")
    ap.add_argument("--limit", type=int, default=0, help="only the first N GEMMs of the workload (profiling)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "mp":
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif is_b2b(args.workload):
        run_b2b(args)
    elif is_conv(args.workload):
        run_conv(args)
    elif args.workload in grouped_names():
        run_grouped(args)
    else:
        run_mp(args)


if __name__ == "__main__":
    main()

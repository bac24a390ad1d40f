"""Cost-model ablation against an exhaustive-search oracle (GPU).

The MikPoly summary (section 5, "cost model effectiveness") compares the
polymerizer with three variants: an oracle that searches the strategies
exhaustively and keeps the fastest program (its search time not counted), a
WAVE variant that minimises the number of waves (large micro-kernels), and a
PIPE variant that maximises the speed of a single pipeline task (small
micro-kernels).  It reports their speed relative to the oracle.

Here, per shape of a workload:

- ``mikpoly``, ``wave`` and ``pipe`` are the plans of the three cost models
  (``mp_set_plan_mode``);
- the oracle runs every Pattern I candidate and the ``--top`` cheapest
  candidates by model cost (``mp_enumerate_plans``), plus the three plans
  above, and keeps the fastest.

Every plan is timed back to back with CUDA events through
``mp_gemm_with_plan``.  The result per variant is sum(T_oracle) / sum(T_variant)
over the workload, together with the host planning time of the heuristic and
of the enumeration.

    python -m micro_polymerization_gb300.ablation [--workload dynamic_sequence] [--top 24] [--count 64] [--analytic]

The cost model is the handle's default (the measured table shipped with the
package); --analytic plans with the analytic model instead.
"""
from __future__ import annotations

import argparse
import json
import sys
import time


def _time_plan(mp, lib, h, plan, ops, reps):
    import ctypes
    import torch
    g, A, B, C, D = ops
    args = (h.ptr, ctypes.byref(plan), g.M, g.N, g.K, A.data_ptr(), g.K, B.data_ptr(), g.N,
            C.data_ptr() if C is not None else None, g.N, D.data_ptr(), g.N, g.alpha, g.beta,
            torch.cuda.current_stream().cuda_stream)
    for _ in range(3):
        st = lib.mp_gemm_with_plan(*args)
        if st != 0:
            raise mp.MPError(st, "mp_gemm_with_plan")
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        lib.mp_gemm_with_plan(*args)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / reps


def _key(p):
    return tuple((r.kernel, r.m0, r.n0, r.m_ext, r.n_ext, r.splits) for r in p.regions())


def run(workload: str = "dynamic_sequence", top: int = 24, count: int = 64, reps: int = 20, device: int = 0,
        analytic: bool = False):
    import torch
    import micro_polymerization_gb300 as mp
    from micro_polymerization_gb300 import workloads as wl

    dev = torch.device("cuda", device)
    torch.cuda.set_device(dev)
    h = mp.mp_init(device, "" if analytic else None)
    lib = mp.library()
    gs = [g for g in wl.workload(workload) if g.batch == 1][:count]
    tot = {"oracle": 0.0, "mikpoly": 0.0, "wave": 0.0, "pipe": 0.0}
    plan_us = enum_us = 0.0
    per_shape = []
    try:
        for i, g in enumerate(gs):
            A, B, C = wl.make_operands(g, device=dev)
            D = torch.empty(g.M, g.N, device=dev)
            ops = (g, A, B, C, D)
            plans = {}
            for name, mode in (("mikpoly", mp.MP_PLAN_MIKPOLY), ("wave", mp.MP_PLAN_WAVE), ("pipe", mp.MP_PLAN_PIPE)):
                mp.mp_set_plan_mode(h, mode)
                t0 = time.perf_counter()
                plans[name] = mp.mp_plan(h, g.M, g.N, g.K)
                if name == "mikpoly":
                    plan_us += (time.perf_counter() - t0) * 1e6
            mp.mp_set_plan_mode(h, mp.MP_PLAN_MIKPOLY)
            t0 = time.perf_counter()
            cands = mp.mp_enumerate_plans(h, g.M, g.N, g.K)
            enum_us += (time.perf_counter() - t0) * 1e6
            pool = {}
            for p in [c for c in cands if c.pattern == 1] + cands[:top] + list(plans.values()):
                pool.setdefault(_key(p), p)
            times = {k: _time_plan(mp, lib, h, p, ops, reps) for k, p in pool.items()}
            t_oracle = min(times.values())
            tot["oracle"] += t_oracle
            row = {"shape": [g.M, g.N, g.K], "oracle_us": round(t_oracle, 2), "candidates": len(pool)}
            for name, p in plans.items():
                t = times[_key(p)]
                tot[name] += t
                row[name + "_us"] = round(t, 2)
            per_shape.append(row)
            del A, B, C, D
    finally:
        h.close()
    n = max(1, len(gs))
    return {
        "workload": workload, "gemms": len(gs), "top": top, "cost_model": "analytic" if analytic else "default",
        "speed_vs_oracle": {k: round(tot["oracle"] / v, 4) for k, v in tot.items() if v > 0},
        "sum_us": {k: round(v, 1) for k, v in tot.items()},
        "plan_us_heuristic": round(plan_us / n, 2), "plan_us_enumeration": round(enum_us / n, 1),
        "per_shape": per_shape,
    }


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--workload", default="dynamic_sequence")
    ap.add_argument("--top", type=int, default=24)
    ap.add_argument("--count", type=int, default=64)
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--device", type=int, default=0)
    ap.add_argument("--per-shape", action="store_true", help="include every shape's times")
    ap.add_argument("--analytic", action="store_true", help="plan with the analytic cost model")
    args = ap.parse_args(argv)
    res = run(args.workload, args.top, args.count, args.reps, args.device, args.analytic)
    if not args.per_shape:
        res.pop("per_shape")
    sys.stdout.write(json.dumps(res) + "\n")
    return 0


if __name__ == "__main__":
    sys.exit(main())

"""Host-side logic of the bench's multi-GPU path, run on CPU with two gloo ranks.

One process per GPU, each with its own copy of the workload (weak scaling);
the only cross-rank operations are the barrier and the max-over-ranks timing
reduction.  No GPU is used here.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as tmp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, l = bench.dist_env()
        out = {"env": [w, r, l]}
        out["max"] = bench.max_over_ranks(1.5 + rank, w)
        bench.barrier(w)
        gs = bench.rank_workload("dynamic_sequence", r)
        out["shapes"] = [[g.M, g.N, g.K] for g in gs]
        out["seeds"] = [g.seed for g in gs]
        one = bench.rank_workload("shape:300,200,100,0.5", r)
        out["one"] = [one[0].M, one[0].N, one[0].K, one[0].beta, one[0].seed]
        q.put((rank, out))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_shapes_not_operands():
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = dict(q.get(timeout=180) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    assert res[0]["env"] == [2, 0, 0] and res[1]["env"] == [2, 1, 1]
    # The timing reduction is a max over ranks.
    assert res[0]["max"] == res[1]["max"] == 2.5
    # Weak scaling: every rank runs the same shapes on its own operands.
    assert res[0]["shapes"] == res[1]["shapes"] and len(res[0]["shapes"]) == 64
    assert all(a != b for a, b in zip(res[0]["seeds"], res[1]["seeds"]))
    assert res[0]["one"][:4] == res[1]["one"][:4] == [300, 200, 100, 0.5]
    assert res[0]["one"][4] != res[1]["one"][4]


def test_reference_arm_other_ranks_exit_without_work():
    """Under torchrun only rank 0 times the oracle; the others exit 0 silently."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1", "--workload", "single_skinny", "--cpu-seconds", "0.5"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["cores"] >= 1

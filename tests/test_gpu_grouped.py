"""GPU parity of the grouped GEMM (mp_gemm_grouped): every problem of a
group against the fp64 oracle under the stated bound, integer data bitwise."""
import numpy as np
import pytest
import torch

import micro_polymerization_gb300 as mp
import oracle
from micro_polymerization_gb300 import workloads as wl

from gpu_util import handle

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _bits(t):
    return wl.bf16_bits(t.cpu())


def _group(shapes, seed, beta=0.5):
    items, host = [], []
    for i, (M, N, K) in enumerate(shapes):
        g = wl.Gemm(M, N, K, alpha=1.0 + 0.25 * (i % 3), beta=beta if i % 2 else 0.0, seed=seed + 7 * i)
        A, B, C = wl.make_operands(g)
        D = torch.full((M, N), float("nan"), device=DEV)
        items.append((A.to(DEV), B.to(DEV), C.to(DEV) if C is not None else None, D, g.alpha, g.beta))
        host.append((A, B, C, g))
    return items, host


def _check_group(items, host):
    torch.cuda.synchronize()
    assert mp.mp_check(handle()) == 0
    probs = [(_bits(A), _bits(B), C.numpy() if C is not None else None, g.alpha, g.beta) for A, B, C, g in host]
    for (D, mag), it, (A, B, C, g) in zip(oracle.gemm_group(probs), items, host):
        ok, worst = oracle.within_bound(it[3].cpu().numpy(), D, mag)
        assert ok, (g, worst)


def test_grouped_ragged_shapes():
    rng = np.random.default_rng(1)
    shapes = [(1, 64, 64), (300, 520, 700), (129, 17, 5), (64, 256, 0), (1000, 96, 33), (7, 1, 130), (255, 384, 256)]
    shapes += [(int(rng.integers(1, 600)), int(rng.integers(1, 600)), int(rng.integers(0, 600))) for _ in range(13)]
    items, host = _group(shapes, seed=11)
    mp.mp_gemm_grouped(handle(), items)
    _check_group(items, host)


def test_grouped_more_than_one_launch():
    rng = np.random.default_rng(2)
    shapes = [(int(rng.integers(1, 300)), int(rng.integers(16, 300)), int(rng.integers(16, 300))) for _ in range(100)]
    items, host = _group(shapes, seed=12)
    mp.mp_gemm_grouped(handle(), items)
    _check_group(items, host)


def test_grouped_unaligned_operands_and_in_place():
    items = []
    host = []
    for i, (M, N, K) in enumerate([(70, 33, 45), (130, 200, 17)]):
        g = wl.Gemm(M, N, K, alpha=1.0, beta=1.0, seed=40 + i)
        A, B, C = wl.make_operands(g)
        # Odd leading dimensions: views into wider buffers.
        Aw = torch.zeros(M, K + 3, dtype=torch.bfloat16, device=DEV)
        Aw[:, :K] = A.to(DEV)
        Dw = C.to(DEV).clone()  # in place: C is D
        items.append((Aw[:, :K], B.to(DEV), Dw, Dw, 1.0, 1.0))
        host.append((A, B, C, g))
    mp.mp_gemm_grouped(handle(), items)
    _check_group(items, host)


def test_grouped_integer_exact():
    shapes = [(100, 70, 129), (33, 300, 64), (257, 64, 200)]
    items, host = [], []
    for i, (M, N, K) in enumerate(shapes):
        A, B, C = wl.integer_operands(M, N, K, seed=50 + i)
        D = torch.empty(M, N, device=DEV)
        items.append((A.to(DEV), B.to(DEV), C.to(DEV), D, 1.0, 1.0))
        host.append((A, B, C))
    mp.mp_gemm_grouped(handle(), items)
    torch.cuda.synchronize()
    for it, (A, B, C) in zip(items, host):
        ref = oracle.gemm(_bits(A), _bits(B), C.numpy(), 1.0, 1.0)
        assert np.array_equal(it[3].cpu().numpy().astype(np.float64), ref)


def test_grouped_experts_workload_sampled():
    """The full grouped_experts workload (48 problems, one call as the bench
    times it), every problem checked on sampled rows against the oracle."""
    gs = wl.grouped_experts()
    rng = np.random.default_rng(3)
    items, host = [], []
    for g in gs:
        A, B, _ = wl.make_operands(g)
        D = torch.full((g.M, g.N), float("nan"), device=DEV)
        items.append((A.to(DEV), B.to(DEV), None, D, g.alpha, g.beta))
        host.append((A, B))
    mp.mp_gemm_grouped(handle(), items)
    torch.cuda.synchronize()
    assert mp.mp_check(handle()) == 0
    for g, it, (A, B) in zip(gs, items, host):
        rows = np.unique(np.concatenate([[0, g.M - 1], rng.integers(0, g.M, 6)]))
        Ab = _bits(A)[rows]
        ref = oracle.gemm(Ab, _bits(B))
        mag = oracle.magnitude(Ab, _bits(B))
        ok, worst = oracle.within_bound(it[3].cpu().numpy()[rows], ref, mag)
        assert ok, (g, worst)

"""mp_gemm_noalloc, the entry point for callers that cannot allocate device
memory (runtimes that own all device memory, pre-reserved memory pools,
loops that must not let an allocation synchronize the device).

It keeps its scratch in a fixed array inside the library instead of a
handle's cudaMalloc'd workspace.  These tests call it through the C ABI twice
in a row -- the second call starts from whatever the first left in the shared
array -- and check both results against the fp64 oracle within the parity
bound used by every GPU test.  The shapes make it use that scratch: split-K
partials and tile counters, and the staging area for unaligned rows.  The
second call must not change the device's free memory.  A bounded wait that
runs out inside one of its kernels is reported by mp_check_noalloc, and the
call after it is correct again.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test.  It passes on its own in a fresh
process as well as after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import micro_polymerization_gb300 as mp
import oracle
from micro_polymerization_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

# The fixed array's limits (csrc/mp_noalloc.cu).
PARTIAL_BYTES = 16 << 20
COUNTERS = 4096

SHAPES = [
    # (M, N, K, alpha, beta): split-K partials + counters
    (105, 1024, 12544, 1.0, 1.0),
    (8, 768, 3072, 1.0, 0.0),
    # rows not 16-byte aligned: staged copies of A and B
    (77, 301, 1001, 1.5, 0.5),
    # no split: plain launch
    (640, 512, 256, 1.0, 0.0),
]


def _call_noalloc(A, B, C, D, alpha, beta):
    lib = mp.library()
    M, K = A.shape
    N = B.shape[1]
    st = lib.mp_gemm_noalloc(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                             C.data_ptr() if C is not None else None, C.stride(0) if C is not None else 0,
                             D.data_ptr(), D.stride(0), ctypes.c_float(alpha), ctypes.c_float(beta),
                             torch.cuda.current_stream().cuda_stream)
    return st


def _oracle(A, B, C, alpha, beta):
    Cn = C.numpy() if C is not None else None
    Ab, Bb = wl.bf16_bits(A), wl.bf16_bits(B)
    return oracle.gemm(Ab, Bb, Cn, alpha, beta), oracle.magnitude(Ab, Bb, Cn, beta)


@pytest.mark.parametrize("M,N,K,alpha,beta", SHAPES)
def test_noalloc_matches_oracle_on_two_calls(M, N, K, alpha, beta):
    dev = torch.device("cuda", 0)
    g = wl.Gemm(M, N, K, alpha=alpha, beta=beta, seed=4242 + M)
    A, B, C = wl.make_operands(g)
    Ad, Bd = A.to(dev), B.to(dev)
    Cd = C.to(dev) if C is not None else None

    if (M, N, K) == (105, 1024, 12544):
        # The shape is chosen to use the split-K scratch.  A regular handle on
        # this device plans with the same cost model and micro-kernel set; its
        # plan splits K and fits the fixed array's partials and counters, so
        # the limits that bind only mp_gemm_noalloc's planner do not change it.
        h = mp.mp_init(0)
        try:
            plan = mp.mp_plan(h, M, N, K)
        finally:
            h.close()
        assert any(r.splits > 1 for r in plan.regions()), "shape chosen to exercise split-K scratch"
        assert plan.workspace_bytes <= PARTIAL_BYTES
        tiles = sum(-(-r.m_ext // r.um) * -(-r.n_ext // r.un) for r in plan.regions() if r.splits > 1)
        assert tiles <= COUNTERS

    Dref, mag = _oracle(A, B, C, alpha, beta)
    for call in range(2):
        D = torch.full((M, N), float("nan"), device=dev)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info(0)[0]
        st = _call_noalloc(Ad, Bd, Cd, D, alpha, beta)
        assert st == mp.MP_OK, mp.mp_status_string(st)
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info(0)[0]
        if call == 1:
            # The first call on a device may load the library's device code
            # (and with it the fixed array); later calls allocate nothing.
            assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
        assert mp.mp_check_noalloc() == mp.MP_OK
        ok, worst = oracle.within_bound(D.cpu().numpy(), Dref, mag)
        assert ok, f"call {call + 1}: outside the parity bound (worst ratio {worst:.3g})"


def test_noalloc_reports_bounded_wait_timeouts():
    """A withheld pipeline stage (hook mode 1), and split-K sums staged in the
    idle operand ring waiting for bytes that never come (mode 2): the kernel
    stops, mp_check_noalloc reports MP_ERR_DEVICE_TIMEOUT and clears the
    status, and the next call matches the oracle."""
    dev = torch.device("cuda", 0)
    g = wl.Gemm(105, 1024, 12544, alpha=1.0, beta=1.0, seed=99)
    A, B, C = wl.make_operands(g)
    Ad, Bd, Cd = A.to(dev), B.to(dev), C.to(dev)
    Dref, mag = _oracle(A, B, C, 1.0, 1.0)
    try:
        for mode in (1, 2):
            D = torch.empty(g.M, g.N, device=dev)
            mp.mp_noalloc_inject_wait_timeout(mode, 50_000_000)  # 50 ms
            assert _call_noalloc(Ad, Bd, Cd, D, 1.0, 1.0) == mp.MP_OK
            assert mp.mp_check_noalloc() == mp.MP_ERR_DEVICE_TIMEOUT, f"mode {mode}"
            assert mp.mp_check_noalloc() == mp.MP_OK
            mp.mp_noalloc_inject_wait_timeout(0, 1_000_000_000)
            D = torch.full((g.M, g.N), float("nan"), device=dev)
            assert _call_noalloc(Ad, Bd, Cd, D, 1.0, 1.0) == mp.MP_OK
            assert mp.mp_check_noalloc() == mp.MP_OK
            ok, worst = oracle.within_bound(D.cpu().numpy(), Dref, mag)
            assert ok, f"after mode {mode}: outside the parity bound (worst ratio {worst:.3g})"
    finally:
        mp.mp_noalloc_inject_wait_timeout(0, 1_000_000_000)


def test_noalloc_rejects_what_its_scratch_cannot_hold():
    """An unaligned operand larger than the 32 MiB staging area is refused
    before anything runs; bad arguments follow mp_gemm's rules."""
    dev = torch.device("cuda", 0)
    M, K, N = 4100, 4097, 8  # A needs 4100 x 4104 bf16 = 33.7 MB once its rows are padded
    A = torch.zeros(M, K, dtype=torch.bfloat16, device=dev)
    B = torch.zeros(K, N, dtype=torch.bfloat16, device=dev)
    D = torch.zeros(M, N, device=dev)
    assert _call_noalloc(A, B, None, D, 1.0, 0.0) == mp.MP_ERR_UNSUPPORTED
    lib = mp.library()
    st = lib.mp_gemm_noalloc(4, 4, 4, A.data_ptr(), 3, B.data_ptr(), 8, None, 0, D.data_ptr(), 8,
                             ctypes.c_float(1.0), ctypes.c_float(0.0), None)
    assert st == mp.MP_ERR_INVALID_ARG  # lda < K

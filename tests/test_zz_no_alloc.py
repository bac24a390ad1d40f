"""mp_gemm_noalloc, the entry point for callers that cannot allocate device
memory (runtimes that own all device memory, pre-reserved memory pools,
loops that must not let an allocation synchronize the device).

It keeps its scratch in a fixed array inside the library instead of a
handle's cudaMalloc'd workspace.  This test calls it through the C ABI twice
in a row -- the second call starts from whatever the first left in the shared
array -- and compares both results with mp_gemm's within the parity bound
used by every GPU test.  The shapes make it use that scratch: split-K
partials and tile counters, and the staging area for unaligned rows.

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


@pytest.mark.parametrize("M,N,K,alpha,beta", SHAPES)
def test_noalloc_matches_mp_gemm_on_two_calls(M, N, K, alpha, beta):
    dev = torch.device("cuda", 0)
    g = wl.Gemm(M, N, K, alpha=alpha, beta=beta, seed=4242 + M)
    A, B, C = wl.make_operands(g)
    Ad, Bd = A.to(dev), B.to(dev)
    Cd = C.to(dev) if C is not None else None

    h = mp.mp_init(0)
    try:
        Dref = torch.empty(M, N, device=dev)
        mp.mp_gemm(h, Ad, Bd, Cd, Dref, alpha, beta)
        torch.cuda.synchronize()
        plan = mp.mp_plan(h, M, N, K)
    finally:
        h.close()
    if (M, N, K) == (105, 1024, 12544):
        assert any(r.splits > 1 for r in plan.regions()), "shape chosen to exercise split-K scratch"

    mag = oracle.magnitude(wl.bf16_bits(A), wl.bf16_bits(B), C.numpy() if C is not None else None, beta)
    for call in range(2):
        D = torch.full((M, N), float("nan"), device=dev)
        st = _call_noalloc(Ad, Bd, Cd, D, alpha, beta)
        assert st == mp.MP_OK, mp.mp_status_string(st)
        torch.cuda.synchronize()
        ok, worst = oracle.within_bound(D.cpu().numpy(), Dref.cpu().numpy().astype(np.float64), mag)
        assert ok, f"call {call + 1}: differs from mp_gemm beyond the bound (worst ratio {worst:.3g})"


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

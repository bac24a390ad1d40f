"""Helpers shared by the GPU parity tests: run the library, compare with the oracle."""
import numpy as np
import torch

import micro_polymerization_gb300 as mp
import oracle
from micro_polymerization_gb300 import workloads as wl

_handle = None


def handle():
    global _handle
    if _handle is None:
        _handle = mp.mp_init(0)
    return _handle


def bits(t):
    return wl.bf16_bits(t)


def run_gemm(A, B, C, alpha, beta, D=None, h=None):
    """A, B bf16 / C fp32 CPU or CUDA tensors; returns D (CPU fp32)."""
    dev = torch.device("cuda", 0)
    Ad, Bd = A.to(dev), B.to(dev)
    Cd = C.to(dev) if C is not None else None
    if D is None:
        D = torch.full((A.shape[0], B.shape[1]), float("nan"), device=dev)
    mp.mp_gemm(h or handle(), Ad, Bd, Cd, D, alpha, beta)
    torch.cuda.synchronize()
    return D.cpu()


def oracle_full(A, B, C, alpha, beta):
    Cn = C.cpu().numpy() if C is not None else None
    return oracle.gemm(bits(A.cpu()), bits(B.cpu()), Cn, alpha, beta), \
        oracle.magnitude(bits(A.cpu()), bits(B.cpu()), Cn, beta)


def assert_parity(D, A, B, C, alpha, beta, what=""):
    Dref, mag = oracle_full(A, B, C, alpha, beta)
    ok, worst = oracle.within_bound(D.numpy(), Dref, mag)
    if not ok:
        err = np.abs(D.numpy().astype(np.float64) - Dref)
        bad = np.argwhere(~(err <= oracle.PARITY_RTOL * mag))
        i, j = bad[0]
        raise AssertionError(
            f"{what}: {len(bad)} entries outside the bound (worst ratio {worst:.3g}); "
            f"first at ({i},{j}): got {D[i, j].item()!r}, want {Dref[i, j]!r}, mag {mag[i, j]!r}")
    return worst


def assert_sampled_parity(D, A, B, C, alpha, beta, rng, n=4096, what=""):
    """Large outputs: every entry of the last row and column tiles, a random
    sample, and a Freivalds probe of the whole matrix."""
    M, N = D.shape
    rows = [rng.integers(0, M, n)]
    cols = [rng.integers(0, N, n)]
    for r0 in (max(0, M - 128), 0):
        rr, cc = np.meshgrid(np.arange(r0, min(M, r0 + 128)), np.arange(max(0, N - 64), N), indexing="ij")
        rows.append(rr.ravel()); cols.append(cc.ravel())
    rr, cc = np.meshgrid(np.arange(max(0, M - 16), M), np.arange(0, min(N, 256)), indexing="ij")
    rows.append(rr.ravel()); cols.append(cc.ravel())
    rows = np.concatenate(rows); cols = np.concatenate(cols)
    Ab, Bb = bits(A.cpu()), bits(B.cpu())
    Cn = C.cpu().numpy() if C is not None else None
    ref, mag = oracle.gemm_entries(Ab, Bb, Cn, alpha, beta, rows, cols)
    got = D.numpy()[rows, cols]
    ok, worst = oracle.within_bound(got, ref, mag)
    assert ok, f"{what}: sampled entries outside the bound (worst ratio {worst:.3g})"
    x = rng.choice([-1.0, 1.0], size=N)
    y, ymag = oracle.freivalds(Ab, Bb, Cn, alpha, beta, D.numpy(), x)
    assert np.all(np.abs(y) <= oracle.PARITY_RTOL * ymag + 1e-30), f"{what}: Freivalds probe failed"
    return worst

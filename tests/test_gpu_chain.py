"""GPU parity of consecutive calls on one stream where a call reads what the
call just before it wrote: its A, its B or its C is the previous call's D.

Each GEMM launch may start while the previous kernel on its stream still
runs, and one-CTA plans warm L2 with their first operand tiles (or, when
beta*C is read, their first C block) before waiting for that kernel.  The
loads that follow the wait must still see every write of the previous
kernel.  Integer-valued data keep every value exact (the bf16 intermediate
too), so each chain must equal the fp64 oracle bit for bit; the buffers are
filled with NaN before every run, so a stale line would show.
"""
import numpy as np
import pytest
import torch

import micro_polymerization_gb300 as mp

from gpu_util import bits, handle, oracle_full

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def ints(rows, cols, seed, lo=-1, hi=1, ld=None):
    """Integer-valued bf16 matrix on the device (a view of a wider one when ld > cols)."""
    g = torch.Generator().manual_seed(seed)
    full = torch.randint(lo, hi + 1, (rows, ld or cols), generator=g).to(torch.bfloat16)
    return full.to(DEV)[:, :cols]


def prefetching_plan(M, N, K):
    """One-CTA regions only, none split or swapped: the plans that prefetch."""
    p = mp.mp_plan(handle(), M, N, K)
    return all(r.splits == 1 and not r.swap and not r.pair for r in p.regions())


def ref_bf16(A, B):
    """The oracle's product of integer operands, as the exact bf16 tensor it is."""
    D, _ = oracle_full(A, B, None, 1.0, 0.0)
    assert np.all(np.abs(D) <= 256.0), "the intermediate must stay exact in bf16"
    return torch.from_numpy(D).to(torch.float32).to(torch.bfloat16)


def assert_exact(D, want, what):
    got = D.cpu().numpy().astype(np.float64)
    bad = np.argwhere(got != want)
    assert len(bad) == 0, f"{what}: {len(bad)} entries differ; first at {tuple(bad[0])}: " \
                          f"got {got[tuple(bad[0])]!r}, want {want[tuple(bad[0])]!r}"


# (M, N, K1, K2): the first GEMM has depth K1 (|sums| <= K1 <= 256 stay exact in
# bf16), the second depth K2.
SHAPES = [(1000, 768, 200, 256), (2048, 3072, 96, 256), (136, 2304, 250, 768)]


@pytest.mark.parametrize("M,N,K1,K2", SHAPES)
def test_a_is_the_previous_calls_output(M, N, K1, K2):
    h = handle()
    A1, B1, B2 = ints(M, K1, 1), ints(K1, K2, 2), ints(K2, N, 3)
    if (M, N) == (1000, 768):
        assert prefetching_plan(M, N, K2)
    D1 = torch.empty(M, K2, device=DEV, dtype=torch.bfloat16)
    D2 = torch.empty(M, N, device=DEV)
    want1 = ref_bf16(A1.cpu(), B1.cpu())
    want2, _ = oracle_full(want1, B2.cpu(), None, 1.0, 0.0)
    for _ in range(3):
        D1.fill_(float("nan"))
        D2.fill_(float("nan"))
        mp.mp_gemm_ex(h, A1, B1, None, D1, 1.0, 0.0)
        mp.mp_gemm(h, D1, B2, None, D2, 1.0, 0.0)
        torch.cuda.synchronize()
        assert np.array_equal(bits(D1.cpu()), bits(want1)), "first GEMM"
        assert_exact(D2, want2, f"A chain {(M, N, K1, K2)}")


@pytest.mark.parametrize("M,N,K1,K2", SHAPES)
def test_b_is_the_previous_calls_output(M, N, K1, K2):
    h = handle()
    A1, B1, A2 = ints(K2, K1, 4), ints(K1, N, 5), ints(M, K2, 6)
    D1 = torch.empty(K2, N, device=DEV, dtype=torch.bfloat16)
    D2 = torch.empty(M, N, device=DEV)
    want1 = ref_bf16(A1.cpu(), B1.cpu())
    want2, _ = oracle_full(A2.cpu(), want1, None, 1.0, 0.0)
    for _ in range(3):
        D1.fill_(float("nan"))
        D2.fill_(float("nan"))
        mp.mp_gemm_ex(h, A1, B1, None, D1, 1.0, 0.0)
        mp.mp_gemm(h, A2, D1, None, D2, 1.0, 0.0)
        torch.cuda.synchronize()
        assert_exact(D2, want2, f"B chain {(M, N, K1, K2)}")


@pytest.mark.parametrize("M,N,K1,K2,ld", [(1000, 768, 200, 256, 768), (1000, 766, 200, 256, 768),
                                          (2048, 3072, 96, 256, 3072), (90, 520, 64, 1024, 520)])
def test_c_is_the_previous_calls_output(M, N, K1, K2, ld):
    """beta*C with C just written by the previous call; N = 766 gives D and C
    rows that are not 16-byte aligned (B's rows are, through a wider view)."""
    h = handle()
    A1, B1 = ints(M, K1, 7, -4, 4), ints(K1, N, 8, ld=ld)
    A2, B2 = ints(M, K2, 9), ints(K2, N, 10, ld=ld)
    if (M, N) == (1000, 768):
        assert prefetching_plan(M, N, K2)
    C = torch.empty(M, N, device=DEV)
    D2 = torch.empty(M, N, device=DEV)
    want1, _ = oracle_full(A1.cpu(), B1.cpu(), None, 1.0, 0.0)
    want2, _ = oracle_full(A2.cpu(), B2.cpu(), torch.from_numpy(want1).float(), 1.0, 0.5)
    for _ in range(3):
        C.fill_(float("nan"))
        D2.fill_(float("nan"))
        mp.mp_gemm(h, A1, B1, None, C, 1.0, 0.0)
        mp.mp_gemm(h, A2, B2, C, D2, 1.0, 0.5)
        torch.cuda.synchronize()
        assert_exact(C, want1, "first GEMM")
        assert_exact(D2, want2, f"C chain {(M, N, K1, K2)}")


def test_in_place_c_is_the_previous_calls_output():
    """D = A2 B2 + 0.5 D in place, where D was written by the call before."""
    h = handle()
    M, N, K1, K2 = 1000, 768, 200, 256
    A1, B1, A2, B2 = ints(M, K1, 11, -4, 4), ints(K1, N, 12), ints(M, K2, 13), ints(K2, N, 14)
    want1, _ = oracle_full(A1.cpu(), B1.cpu(), None, 1.0, 0.0)
    want2, _ = oracle_full(A2.cpu(), B2.cpu(), torch.from_numpy(want1).float(), 1.0, 0.5)
    D = torch.empty(M, N, device=DEV)
    for _ in range(3):
        D.fill_(float("nan"))
        mp.mp_gemm(h, A1, B1, None, D, 1.0, 0.0)
        mp.mp_gemm(h, A2, B2, D, D, 1.0, 0.5)
        torch.cuda.synchronize()
        assert_exact(D, want2, "in-place chain")


def test_conv_input_is_the_previous_calls_output():
    """mp_conv2d whose X (NHWC) the previous call wrote as a bf16 GEMM output."""
    import oracle
    h = handle()
    N, H, W, C, K, R, S = 4, 20, 20, 64, 128, 3, 3
    A1, B1 = ints(N * H * W, 200, 15), ints(200, C, 16)
    F = ints(R * S * C, K, 17).reshape(R, S, C, K)
    Xbuf = torch.empty(N * H * W, C, device=DEV, dtype=torch.bfloat16)
    D = torch.empty(N, H, W, K, device=DEV)
    want_x = ref_bf16(A1.cpu(), B1.cpu())
    want = oracle.conv2d_nhwc(bits(want_x.reshape(N, H, W, C)), bits(F.cpu()), None, 1.0, 0.0, 1, 1)
    for _ in range(3):
        Xbuf.fill_(float("nan"))
        D.fill_(float("nan"))
        mp.mp_gemm_ex(h, A1, B1, None, Xbuf, 1.0, 0.0)
        mp.mp_conv2d(h, Xbuf.view(N, H, W, C), F, None, D, 1.0, 0.0, 1, 1)
        torch.cuda.synchronize()
        assert mp.mp_check(h) == 0
        assert_exact(D.reshape(-1, K), want.reshape(-1, K), "conv chain")


def test_fused_pair_input_is_the_previous_calls_output():
    """mp_gemm_b2b (fused form) whose A0 the previous call wrote as a bf16
    GEMM output; entries of A0 in {-1, 0, 1} keep the on-chip bf16 D0 exact."""
    import oracle
    h = handle()
    M, K0, N0, N1 = 1000, 192, 256, 768
    A1 = ints(M, 8, 18)
    B1 = torch.zeros(8, K0, dtype=torch.bfloat16)
    B1[0] = ints(1, K0, 19).cpu()[0]
    B1 = B1.to(DEV)
    W0, W1 = ints(K0, N0, 20), ints(N0, N1, 21)
    A0 = torch.empty(M, K0, device=DEV, dtype=torch.bfloat16)
    D1 = torch.empty(M, N1, device=DEV)
    want_a0 = ref_bf16(A1.cpu(), B1.cpu())
    want, _ = oracle.b2b(bits(want_a0), bits(W0.cpu()), None, bits(W1.cpu()), None, 1.0, 0.0, 1.0, 0.0, 1)
    mp.mp_set_b2b_mode(h, mp.MP_B2B_FUSED)
    try:
        for _ in range(3):
            A0.fill_(float("nan"))
            D1.fill_(float("nan"))
            mp.mp_gemm_ex(h, A1, B1, None, A0, 1.0, 0.0)
            mp.mp_gemm_b2b(h, A0, W0, None, W1, None, D1, 1.0, 0.0, 1.0, 0.0, 1)
            torch.cuda.synchronize()
            assert mp.mp_check(h) == 0
            assert_exact(D1, want, "fused pair chain")
    finally:
        mp.mp_set_b2b_mode(h, mp.MP_B2B_AUTO)

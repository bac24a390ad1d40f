"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Bound (bf16 inputs, fp32 accumulation, fp32 output), element by element:
    |D - D_ref| <= 2e-3 * (sum_k |A_ik||B_kj| + |beta*C_ij|)
Integer-valued inputs make every fp32 partial sum exact, so there the GPU
result must equal the oracle bit for bit, whatever the tile order or split-K.
"""
import itertools

import numpy as np
import pytest
import torch

import micro_polymerization_gb300 as mp
from micro_polymerization_gb300 import workloads as wl

from gpu_util import assert_parity, assert_sampled_parity, handle, oracle_full, run_gemm

pytestmark = pytest.mark.gpu


def rand_problem(M, N, K, seed, beta=0.0):
    g = wl.Gemm(M, N, K, alpha=1.0, beta=beta, seed=seed)
    return wl.make_operands(g)


# --------------------------------------------------------------------------
# small shapes: brute force over every combination of tiny sizes
# --------------------------------------------------------------------------
TINY = list(range(1, 10))  # every combination of sizes 1..9


def test_tiny_shapes_bruteforce():
    for M, N, K in itertools.product(TINY, TINY, TINY):
        A, B, C = rand_problem(M, N, K, seed=M * 100 + N * 10 + K, beta=0.5)
        D = run_gemm(A, B, C, 1.5, 0.5)
        assert_parity(D, A, B, C, 1.5, 0.5, what=f"{(M, N, K)}")


EDGE = [1, 15, 16, 17, 63, 64, 65, 127, 128, 129, 255, 257]


@pytest.mark.parametrize("M", EDGE)
def test_edge_shapes_integer_exact(M):
    """Tile edges in M, N and K with integer data: bitwise equal to the oracle."""
    rng = np.random.default_rng(M)
    for N in rng.choice(EDGE, 4, replace=False):
        for K in rng.choice([1, 63, 64, 65, 128, 129, 300], 2, replace=False):
            A, B, C = wl.integer_operands(M, int(N), int(K), seed=int(M * 7 + N * 3 + K))
            D = run_gemm(A, B, C, 1.0, 1.0)
            Dref, _ = oracle_full(A, B, C, 1.0, 1.0)
            assert np.array_equal(D.numpy().astype(np.float64), Dref), (M, N, K)


def test_identity_b_gives_a_exactly():
    for M, K in [(1, 64), (100, 128), (129, 200), (300, 72)]:
        A, _, _ = rand_problem(M, K, K, seed=M + K)
        eye = torch.eye(K, dtype=torch.bfloat16)
        D = run_gemm(A, eye, None, 1.0, 0.0)
        assert torch.equal(D, A.float()), (M, K)


def test_permutation_b_permutes_columns():
    M, K = 77, 136
    A, _, _ = rand_problem(M, K, K, seed=3)
    perm = torch.randperm(K, generator=torch.Generator().manual_seed(1))
    P = torch.zeros(K, K, dtype=torch.bfloat16)
    P[perm, torch.arange(K)] = 1
    D = run_gemm(A, P, None, 1.0, 0.0)
    assert torch.equal(D, A.float()[:, perm])


def test_closed_form_ones():
    for M, N, K in [(33, 70, 129), (5, 300, 1000), (200, 17, 64)]:
        A = torch.ones(M, K, dtype=torch.bfloat16)
        B = torch.ones(K, N, dtype=torch.bfloat16)
        C = torch.arange(M * N, dtype=torch.float32).reshape(M, N) % 7
        D = run_gemm(A, B, C, 1.5, 0.5)
        assert torch.equal(D, 1.5 * K + 0.5 * C), (M, N, K)


# --------------------------------------------------------------------------
# every micro-kernel of the set, with and without split-K
# --------------------------------------------------------------------------
def _kernels():
    hw, ks = mp.mp_get_hw(handle())
    return ks


@pytest.mark.parametrize("splits", [1, 3])
def test_each_micro_kernel(splits):
    h = handle()
    ks = _kernels()
    try:
        for k, desc in enumerate(ks):
            if desc.pair and splits > 1:
                continue  # CTA pairs do not split K
            for (M, N, K) in [(200, 300, 500), (37, 520, 130), (130, 129, 64)]:
                mp.mp_force_plan(h, k, splits)
                A, B, C = rand_problem(M, N, K, seed=k * 31 + M, beta=0.5)
                D = run_gemm(A, B, C, 1.5, 0.5)
                assert_parity(D, A, B, C, 1.5, 0.5,
                              what=f"kernel {k} ({desc.um}x{desc.un} swap={desc.swap}) splits={splits} {(M, N, K)}")
    finally:
        mp.mp_force_plan(h, -1, 0)


@pytest.mark.parametrize("M,N,K", [(421, 1000, 320), (256, 512, 640), (1000, 768, 200), (128, 2304, 768),
                                   (2048, 1024, 1024)])
def test_pair_kernels_match_single_cta_kernels_and_oracle(M, N, K):
    """A 256-row tile on a CTA pair (pair MMA, each CTA holding half of A's
    rows and of B's columns) computes exactly what two 128-row tiles on one
    CTA each compute: the same MMAs per output row, so the outputs agree bit
    for bit.  Odd tile-row counts leave the second half of the last pair past
    the end of D."""
    h = _handle_with_pair192()
    try:
        _, ks = mp.mp_get_hw(h)
        pairs = [(k, d) for k, d in enumerate(ks) if d.pair]
        assert {(d.um, d.un) for _, d in pairs} == {(256, 256), (256, 192), (256, 128)}
        for k, d in pairs:
            single = next(i for i, e in enumerate(ks) if not e.pair and not e.swap and e.un == d.un)
            A, B, C = rand_problem(M, N, K, seed=k * 7 + M, beta=0.5)
            mp.mp_force_plan(h, single, 1)
            D1 = run_gemm(A, B, C, 1.25, 0.5, h=h)
            mp.mp_force_plan(h, k, 1)
            D2 = run_gemm(A, B, C, 1.25, 0.5, h=h)
            assert torch.equal(D1, D2), f"pair kernel {k} ({d.um}x{d.un}) {(M, N, K)}"
            assert_parity(D2, A, B, C, 1.25, 0.5, what=f"pair kernel {k} {(M, N, K)}")
    finally:
        h.close()


def _handle_with_pair192():
    """A handle whose set includes the 256 x 192 pair (opt-in: MP_PAIR192=1)."""
    import os
    os.environ["MP_PAIR192"] = "1"
    try:
        return mp.mp_init(0)
    finally:
        del os.environ["MP_PAIR192"]


def test_pair192_is_opt_in_and_matches_oracle_on_every_edge():
    """The 256 x 192 pair (each CTA holding 96 columns of B with the 64-byte
    swizzle) is left out of the default set and joins it with MP_PAIR192=1,
    after the other kernels.  Ragged rows and columns (a last pair half past M,
    a CTA's 96 columns past N, wholly or partly), beta * C, and a K loop not a
    multiple of 64."""
    ks_default = _kernels()
    assert not any(d.pair and d.un == 192 for d in ks_default)
    h = _handle_with_pair192()
    try:
        _, ks = mp.mp_get_hw(h)
        assert [(d.um, d.un, d.swap, d.pair) for d in ks[:len(ks_default)]] == \
               [(d.um, d.un, d.swap, d.pair) for d in ks_default]
        k = next(i for i, d in enumerate(ks) if d.pair and d.un == 192)
        for (M, N, K) in [(300, 520, 700), (129, 97, 65), (700, 192 * 3, 1000), (513, 1000, 333)]:
            mp.mp_force_plan(h, k, 1)
            A, B, C = rand_problem(M, N, K, seed=M + N, beta=0.5)
            D = run_gemm(A, B, C, 1.5, 0.5, h=h)
            assert_parity(D, A, B, C, 1.5, 0.5, what=f"pair 256x192 {(M, N, K)}")
    finally:
        h.close()


def test_pair_kernel_launches_as_cluster(capfd):
    """A plan of pair tiles launches as two-CTA clusters (the plan log says so)."""
    import os
    os.environ["MP_LOG"] = "1"
    try:
        h = mp.mp_init(0)
    finally:
        del os.environ["MP_LOG"]
    try:
        ks = _kernels()
        k = next(i for i, d in enumerate(ks) if d.pair and d.un == 256)
        mp.mp_force_plan(h, k, 1)
        A, B, C = rand_problem(1024, 1024, 256, seed=3)
        D = run_gemm(A, B, None, 1.0, 0.0, h=h)
        err = capfd.readouterr().err
        assert "cluster=2" in err, err
        assert_parity(D, A, B, None, 1.0, 0.0, what="pair 1024^2 x 256")
    finally:
        h.close()


def test_handle_without_pairs_drops_pair_kernels():
    """MP_PAIR=0 when the handle is made: no pair micro-kernels in its set,
    and the other kernels keep their indices."""
    import os
    os.environ["MP_PAIR"] = "0"
    try:
        h = mp.mp_init(0)
    finally:
        del os.environ["MP_PAIR"]
    try:
        _, ks0 = mp.mp_get_hw(h)
        ks = _kernels()
        assert not any(d.pair for d in ks0)
        assert [(d.um, d.un, d.swap) for d in ks0] == [(d.um, d.un, d.swap) for d in ks if not d.pair]
        A, B, C = rand_problem(300, 1000, 500, seed=4)
        assert_parity(run_gemm(A, B, None, 1.0, 0.0, h=h), A, B, None, 1.0, 0.0, what="no-pair handle")
    finally:
        h.close()


def test_split_k_integer_exact_and_deterministic():
    h = handle()
    A, B, C = wl.integer_operands(105, 1024, 4000, seed=9)
    try:
        for k, desc in enumerate(_kernels()):
            mp.mp_force_plan(h, k, 1 if desc.pair else 7)
            D1 = run_gemm(A, B, C, 1.0, 1.0)
            D2 = run_gemm(A, B, C, 1.0, 1.0)
            Dref, _ = oracle_full(A, B, C, 1.0, 1.0)
            assert np.array_equal(D1.numpy().astype(np.float64), Dref), k
            assert torch.equal(D1, D2)
    finally:
        mp.mp_force_plan(h, -1, 0)


def _handle_with(env):
    """A handle made with extra environment settings (read at creation)."""
    import os
    old = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        return mp.mp_init(0)
    finally:
        for k, v in old.items():
            if v is None:
                del os.environ[k]
            else:
                os.environ[k] = v


@pytest.mark.parametrize("M,N,K,splits", [(105, 1024, 4000, 4), (300, 517, 2000, 3), (37, 520, 1300, 8),
                                          (105, 1024, 12544, 16)])
def test_split_k_on_chip_matches_global_bitwise(M, N, K, splits, capfd):
    """Split-K reduced on chip (a cluster of S CTAs summing through
    distributed shared memory) and through the global workspace add the same
    partials in the same split order: bit-identical outputs, within the bound."""
    hg = _handle_with({"MP_CSPLIT": "0"})
    hc = _handle_with({"MP_LOG": "1"})
    A, B, C = rand_problem(M, N, K, seed=M + splits, beta=0.5)
    try:
        for k, desc in enumerate(_kernels()):
            if desc.pair:
                continue
            mp.mp_force_plan(hg, k, splits)
            mp.mp_force_plan(hc, k, splits)
            capfd.readouterr()
            Dc = run_gemm(A, B, C, 1.5, 0.5, h=hc)
            log = capfd.readouterr().err
            Dg = run_gemm(A, B, C, 1.5, 0.5, h=hg)
            p = mp.mp_plan(hc, M, N, K)
            s_eff = p.region[0].splits
            tasks = sum(r.f_parallel for r in p.regions())
            if s_eff <= 8 and tasks <= 64:  # portable cluster sizes: surely one wave
                assert f"cluster={s_eff}" in log, (k, log)
            assert torch.equal(Dc, Dg), f"kernel {k} ({desc.um}x{desc.un} swap={desc.swap}) {(M, N, K)} S={s_eff}"
            assert_parity(Dc, A, B, C, 1.5, 0.5, what=f"on-chip split kernel {k} {(M, N, K)} S={s_eff}")
    finally:
        hg.close()
        hc.close()


def test_repeat_runs_bitwise_equal():
    A, B, C = rand_problem(105, 1024, 12544, seed=1000, beta=1.0)
    D1 = run_gemm(A, B, C, 1.0, 1.0)
    D2 = run_gemm(A, B, C, 1.0, 1.0)
    assert torch.equal(D1, D2)


# --------------------------------------------------------------------------
# layouts: padded and unaligned leading dimensions, offset pointers, in place
# --------------------------------------------------------------------------
def test_padded_leading_dimensions():
    dev = torch.device("cuda", 0)
    M, N, K = 150, 200, 260
    A, B, C = rand_problem(M, N, K, seed=11, beta=0.5)
    Ap = torch.zeros(M, K + 24, dtype=torch.bfloat16); Ap[:, :K] = A
    Bp = torch.zeros(K, N + 40, dtype=torch.bfloat16); Bp[:, :N] = B
    Cp = torch.zeros(M, N + 8); Cp[:, :N] = C
    Dp = torch.full((M, N + 12), 7.0, device=dev)
    mp.mp_gemm(handle(), Ap.to(dev)[:, :K], Bp.to(dev)[:, :N], Cp.to(dev)[:, :N], Dp[:, :N], 1.5, 0.5)
    torch.cuda.synchronize()
    Dp = Dp.cpu()
    assert torch.all(Dp[:, N:] == 7.0), "write past the row end"
    assert_parity(Dp[:, :N].contiguous(), A, B, C, 1.5, 0.5, what="padded ld")


@pytest.mark.parametrize("M,N,K", [(31, 45, 77), (130, 257, 1001), (5, 1023, 333), (300, 9, 12001)])
def test_unaligned_rows_are_repacked(M, N, K):
    """Dense odd leading dimensions (rows not 16-byte aligned)."""
    A, B, C = rand_problem(M, N, K, seed=M + N + K, beta=0.5)
    D = run_gemm(A, B, C, 1.5, 0.5)
    assert_parity(D, A, B, C, 1.5, 0.5, what=f"unaligned {(M, N, K)}")


@pytest.mark.parametrize("beta", [0.5, 0.0])
@pytest.mark.parametrize("splits", [1, 3])
def test_unaligned_d_rows_every_kernel(splits, beta):
    """D whose row pitch is not 16-byte aligned (odd leading dimension): the
    row-wise epilogue and split-K reduction, for every micro-kernel, with
    and without beta * C, and canaries in the padding of each row."""
    dev = torch.device("cuda", 0)
    h = handle()
    M, N, K, ldd = 300, 517, 200, 523
    A, B, C = rand_problem(M, N, K, seed=21, beta=0.5)
    try:
        for k, desc in enumerate(_kernels()):
            if desc.pair and splits > 1:
                continue
            mp.mp_force_plan(h, k, splits)
            buf = torch.full((M * ldd,), -777.0, device=dev)
            D = buf.view(M, ldd)[:, :N]
            mp.mp_gemm(h, A.to(dev), B.to(dev), C.to(dev), D, 1.5, beta)
            torch.cuda.synchronize()
            full = buf.view(M, ldd).cpu()
            assert torch.all(full[:, N:] == -777.0), f"kernel {k}: write past the row end"
            assert_parity(full[:, :N].contiguous(), A, B, C, 1.5, beta,
                          what=f"unaligned D kernel {k} ({desc.um}x{desc.un} swap={desc.swap}) "
                               f"splits={splits} beta={beta}")
    finally:
        mp.mp_force_plan(h, -1, 0)


def test_offset_base_pointers():
    dev = torch.device("cuda", 0)
    M, N, K = 70, 96, 128
    A, B, C = rand_problem(M, N, K, seed=5, beta=0.5)
    Abuf = torch.zeros(M * K + 3, dtype=torch.bfloat16, device=dev)
    Bbuf = torch.zeros(K * N + 5, dtype=torch.bfloat16, device=dev)
    Aview = Abuf[1:1 + M * K].view(M, K); Aview.copy_(A.to(dev))
    Bview = Bbuf[3:3 + K * N].view(K, N); Bview.copy_(B.to(dev))
    D = torch.empty(M, N, device=dev)
    mp.mp_gemm(handle(), Aview, Bview, C.to(dev), D, 1.5, 0.5)
    torch.cuda.synchronize()
    assert_parity(D.cpu(), A, B, C, 1.5, 0.5, what="offset pointers")


def test_in_place_c_equals_d():
    dev = torch.device("cuda", 0)
    A, B, C = rand_problem(129, 140, 200, seed=8, beta=0.5)
    CD = C.to(dev).clone()
    mp.mp_gemm(handle(), A.to(dev), B.to(dev), CD, CD, 1.5, 0.5)
    torch.cuda.synchronize()
    assert_parity(CD.cpu(), A, B, C, 1.5, 0.5, what="in place")


@pytest.mark.parametrize("splits", [1, 3])
def test_in_place_every_micro_kernel(splits):
    """C = D in place with every micro-kernel forced: each epilogue path reads
    an element of C before it writes that element of D (the swapped tiles
    read a column's 16 values of C before their 16 stores)."""
    h = handle()
    dev = torch.device("cuda", 0)
    try:
        for k, desc in enumerate(_kernels()):
            if desc.pair and splits > 1:
                continue
            for (M, N, K) in [(37, 520, 130), (130, 129, 64), (19, 200, 300)]:
                mp.mp_force_plan(h, k, splits)
                A, B, C = rand_problem(M, N, K, seed=k * 17 + N, beta=0.5)
                CD = C.to(dev).clone()
                mp.mp_gemm(h, A.to(dev), B.to(dev), CD, CD, 1.5, 0.5)
                torch.cuda.synchronize()
                assert_parity(CD.cpu(), A, B, C, 1.5, 0.5,
                              what=f"in place, kernel {k} ({desc.um}x{desc.un} swap={desc.swap}) splits={splits} {(M, N, K)}")
    finally:
        mp.mp_force_plan(h, -1, 0)


def test_k_zero_and_empty():
    dev = torch.device("cuda", 0)
    C = torch.randn(33, 65)
    A = torch.empty(33, 0, dtype=torch.bfloat16)
    B = torch.empty(0, 65, dtype=torch.bfloat16)
    D = torch.full((33, 65), float("nan"), device=dev)
    mp.mp_gemm(handle(), A.to(dev), B.to(dev), C.to(dev), D, 2.0, 0.5)
    torch.cuda.synchronize()
    assert torch.equal(D.cpu(), 0.5 * C)
    E = torch.full((0, 5), 1.0, device=dev)
    mp.mp_gemm(handle(), torch.empty(0, 7, dtype=torch.bfloat16, device=dev),
               torch.empty(7, 5, dtype=torch.bfloat16, device=dev), None, E, 1.0, 0.0)


def test_output_guard_bands():
    """Nothing is written outside D: canaries before, after and between rows."""
    dev = torch.device("cuda", 0)
    M, N, K, pad = 133, 250, 96, 64
    A, B, _ = rand_problem(M, N, K, seed=12)
    buf = torch.full((pad + M * (N + 3) + pad,), -12345.0, device=dev)
    D = buf[pad:pad + M * (N + 3)].view(M, N + 3)[:, :N]
    for k, desc in enumerate(_kernels()):
        mp.mp_force_plan(handle(), k, 1 if desc.pair else 2)
        mp.mp_gemm(handle(), A.to(dev), B.to(dev), None, D, 1.0, 0.0)
    mp.mp_force_plan(handle(), -1, 0)
    torch.cuda.synchronize()
    b = buf.cpu()
    assert torch.all(b[:pad] == -12345.0) and torch.all(b[-pad:] == -12345.0)
    assert torch.all(b[pad:pad + M * (N + 3)].view(M, N + 3)[:, N:] == -12345.0)


# --------------------------------------------------------------------------
# merged GEMMs (shared operand concat; same-shape batch)
# --------------------------------------------------------------------------
def test_shared_operand_merge_equals_separate():
    """A x concat(Wq, Wk, Wv) == concat(A Wq, A Wk, A Wv), bitwise on integers."""
    A, B, _ = wl.integer_operands(257, 3 * 320, 256, seed=21)
    merged = run_gemm(A, B, None, 1.0, 0.0)
    parts = [run_gemm(A, B[:, i * 320:(i + 1) * 320].contiguous(), None, 1.0, 0.0) for i in range(3)]
    assert torch.equal(merged, torch.cat(parts, dim=1))


@pytest.mark.parametrize("seq", [16, 100, 257])
def test_batched_equals_loop(seq):
    dev = torch.device("cuda", 0)
    g = wl.Gemm(seq, seq, 64, batch=12, seed=seq)
    A, B, _ = wl.make_operands(g)
    D = torch.empty(12, seq, seq, device=dev)
    mp.mp_gemm_batched(handle(), A.to(dev), B.to(dev), None, D, 1.0, 0.0)
    torch.cuda.synchronize()
    D = D.cpu()
    for b in range(12):
        assert_parity(D[b], A[b], B[b], None, 1.0, 0.0, what=f"batch {b}")
    Ai, Bi, _ = wl.integer_operands(seq, seq, 64, seed=seq)
    Ab = torch.stack([Ai] * 3); Bb = torch.stack([Bi, -Bi, Bi])
    Db = torch.empty(3, seq, seq, device=dev)
    mp.mp_gemm_batched(handle(), Ab.to(dev), Bb.to(dev), None, Db, 1.0, 0.0)
    torch.cuda.synchronize()
    single = run_gemm(Ai, Bi, None, 1.0, 0.0)
    assert torch.equal(Db[0].cpu(), single) and torch.equal(Db[1].cpu(), -single)


@pytest.mark.parametrize("M,N,K", [(37, 45, 77), (130, 9, 263)])
def test_batched_unaligned_rows_are_repacked(M, N, K):
    """Batched operands whose rows and batch strides are not 16-byte
    aligned (odd K and N): both are staged in one copy, and a broadcast A
    (batch stride 0) is staged once."""
    dev = torch.device("cuda", 0)
    g = wl.Gemm(M, N, K, batch=5, beta=0.5, seed=M + K)
    A, B, C = wl.make_operands(g)
    D = torch.empty(5, M, N, device=dev)
    mp.mp_gemm_batched(handle(), A.to(dev), B.to(dev), C.to(dev), D, 1.5, 0.5)
    torch.cuda.synchronize()
    D = D.cpu()
    for b in range(5):
        assert_parity(D[b], A[b], B[b], C[b], 1.5, 0.5, what=f"unaligned batch {b} {(M, N, K)}")
    D2 = torch.empty(5, M, N, device=dev)
    mp.mp_gemm_batched(handle(), A[:1].to(dev), B.to(dev), None, D2, 1.0, 0.0)
    torch.cuda.synchronize()
    D2 = D2.cpu()
    for b in range(5):
        assert_parity(D2[b], A[0], B[b], None, 1.0, 0.0, what=f"broadcast A, batch {b}")


@pytest.mark.parametrize("lda_extra,ldb_extra", [(0, 0), (1, 3)])
def test_operands_two_bytes_past_a_word(lda_extra, ldb_extra):
    """A and B start 2 bytes past a 4-byte boundary: with an even row pitch
    every row starts there, with an odd one every other row does."""
    dev = torch.device("cuda", 0)
    M, N, K = 67, 90, 150
    A, B, C = rand_problem(M, N, K, seed=9, beta=0.5)
    lda, ldb = K + lda_extra, N + ldb_extra
    Abuf = torch.zeros(1 + M * lda + 8, dtype=torch.bfloat16, device=dev)
    Bbuf = torch.zeros(1 + K * ldb + 8, dtype=torch.bfloat16, device=dev)
    Av = Abuf[1:1 + M * lda].view(M, lda)[:, :K]
    Bv = Bbuf[1:1 + K * ldb].view(K, ldb)[:, :N]
    Av.copy_(A.to(dev))
    Bv.copy_(B.to(dev))
    assert Av.data_ptr() % 4 == 2 and Bv.data_ptr() % 4 == 2
    D = torch.empty(M, N, device=dev)
    mp.mp_gemm(handle(), Av, Bv, C.to(dev), D, 1.5, 0.5)
    torch.cuda.synchronize()
    assert_parity(D.cpu(), A, B, C, 1.5, 0.5, what=f"2-byte offset, ld +{lda_extra}/+{ldb_extra}")


def test_batched_shared_operand_stride_zero():
    dev = torch.device("cuda", 0)
    A, B, _ = rand_problem(64, 80, 96, seed=4)
    Bs = torch.stack([B, 2 * B, -B])
    D = torch.empty(3, 64, 80, device=dev)
    mp.mp_gemm_batched(handle(), A.to(dev).unsqueeze(0), Bs.to(dev), None, D, 1.0, 0.0)
    torch.cuda.synchronize()
    for b in range(3):
        assert_parity(D[b].cpu(), A, Bs[b], None, 1.0, 0.0, what=f"shared A, batch {b}")


# --------------------------------------------------------------------------
# the workloads at full size (sampled where the oracle cannot do all of it)
# --------------------------------------------------------------------------
def test_single_skinny_full_oracle():
    g = wl.single_skinny()[0]
    A, B, C = wl.make_operands(g)
    D = run_gemm(A, B, C, g.alpha, g.beta)
    assert_parity(D, A, B, C, g.alpha, g.beta, what="(105,1024,12544)")


@pytest.mark.parametrize("name,count", [("dynamic_sequence", 6), ("dynamic_resolution", 4),
                                        ("merged_qkv", 4), ("stress", 12)])
def test_workload_samples_full_size(name, count):
    rng = np.random.default_rng(len(name))
    shapes = wl.workload(name)
    picks = [shapes[i] for i in rng.choice(len(shapes), count, replace=False)]
    if name == "stress":
        picks.append(shapes[-1])  # 4096^3
    dev = torch.device("cuda", 0)
    for g in picks:
        A, B, C = wl.make_operands(g, device=dev)
        D = torch.empty(g.M, g.N, device=dev)
        mp.mp_gemm(handle(), A, B, C, D, g.alpha, g.beta)
        torch.cuda.synchronize()
        assert_sampled_parity(D.cpu(), A.cpu(), B.cpu(), C.cpu() if C is not None else None,
                              g.alpha, g.beta, rng, what=f"{name} {(g.M, g.N, g.K)}")


@pytest.mark.parametrize("M,N,K,alpha,beta", [(6144, 6144, 6144, 1.0, 0.0), (10332, 13649, 4045, 1.5, 0.5)])
def test_large_pair_plans_in_grouped_order(M, N, K, alpha, beta):
    """Large problems: CTA-pair micro-kernels, tiles handed out in groups of
    tile rows (the operands do not fit L2), with aligned D and with unaligned
    D plus beta * C."""
    h = handle()
    _, ks = mp.mp_get_hw(h)
    p = mp.mp_plan(h, M, N, K)
    if any(d.pair for d in ks):
        assert all(r.pair for r in p.regions()), [(r.um, r.un, r.pair) for r in p.regions()]
    dev = torch.device("cuda", 0)
    g = wl.Gemm(M, N, K, alpha=alpha, beta=beta, seed=M % 97)
    A, B, C = wl.make_operands(g, device=dev)
    D = torch.empty(M, N, device=dev)
    mp.mp_gemm(h, A, B, C, D, alpha, beta)
    torch.cuda.synchronize()
    rng = np.random.default_rng(M)
    assert_sampled_parity(D.cpu(), A.cpu(), B.cpu(), C.cpu() if C is not None else None, alpha, beta, rng,
                          what=f"large {(M, N, K)}")


@pytest.mark.parametrize("M,N,K", [(300, 520, 700), (1000, 768, 1300), (129, 2304, 4096)])
def test_explicit_plans_and_ablation_models_match_oracle(M, N, K):
    """Any candidate of the search space (cheap or expensive, Pattern I or
    II, split or not) run through mp_gemm_with_plan, and the plans of the
    WAVE and PIPE cost models, compute the same D within the bound."""
    h = handle()
    dev = torch.device("cuda", 0)
    A, B, C = rand_problem(M, N, K, seed=M + 3, beta=0.5)
    Ad, Bd, Cd = A.to(dev), B.to(dev), C.to(dev)
    cands = mp.mp_enumerate_plans(h, M, N, K)
    two = [c for c in cands if c.pattern == 2]
    mid = len(cands) // 2
    picks = cands[:3] + two[:2] + two[len(two) // 2:len(two) // 2 + 1] + cands[mid:mid + 2] + cands[-2:]
    for p in picks:
        D = torch.full((M, N), float("nan"), device=dev)
        mp.mp_gemm_with_plan(h, p, Ad, Bd, Cd, D, 1.5, 0.5)
        torch.cuda.synchronize()
        desc = [(r.um, r.un, r.swap, r.pair, r.splits, r.m0, r.n0, r.m_ext, r.n_ext) for r in p.regions()]
        assert_parity(D.cpu(), A, B, C, 1.5, 0.5, what=f"plan {desc}")
    try:
        for mode in (mp.MP_PLAN_WAVE, mp.MP_PLAN_PIPE):
            mp.mp_set_plan_mode(h, mode)
            assert_parity(run_gemm(A, B, C, 1.5, 0.5), A, B, C, 1.5, 0.5, what=f"mode {mode}")
    finally:
        mp.mp_set_plan_mode(h, mp.MP_PLAN_MIKPOLY)
    # Regions that overlap are refused before anything runs.
    bad = mp.MpPlanInfo()
    bad.num_regions = 2
    for i, (m0, me) in enumerate([(0, M // 2 + 8), (M // 2, M - M // 2)]):
        bad.region[i].kernel, bad.region[i].m0, bad.region[i].m_ext = 0, m0, me
        bad.region[i].n0, bad.region[i].n_ext, bad.region[i].splits = 0, N, 1
    with pytest.raises(mp.MPError) as e:
        mp.mp_gemm_with_plan(h, bad, Ad, Bd, Cd, torch.empty(M, N, device=dev), 1.5, 0.5)
    assert e.value.status == mp.MP_ERR_PLAN


@pytest.mark.parametrize("M,N,K,beta", [(300, 520, 700, 0.5), (300, 517, 450, 0.5), (130, 517, 200, 0.0),
                                        (300, 520, 700, 0.0)])
def test_epilogue_variants_every_kernel(M, N, K, beta):
    """mp_gemm_ex: ReLU / GELU on alpha*A*B + beta*C and fp32 / bf16 D, for
    every micro-kernel with and without split-K, on aligned and odd-pitch D:
    within the bound carried through the activation (plus one bf16 unit of
    the reference for bf16 D)."""
    import oracle
    h = handle()
    dev = torch.device("cuda", 0)
    A, B, C = rand_problem(M, N, K, seed=M + N, beta=beta)
    Dref, mag = oracle_full(A, B, C, 1.25, beta)
    Ad, Bd = A.to(dev), B.to(dev)
    Cd = C.to(dev) if C is not None else None
    refs = {act: oracle.epilogue(Dref, act) for act in (mp.MP_ACT_NONE, mp.MP_ACT_RELU, mp.MP_ACT_GELU)}
    try:
        for k, desc in enumerate(_kernels()):
            for splits in ((1,) if desc.pair else (1, 3)):
                mp.mp_force_plan(h, k, splits)
                for act, ref in refs.items():
                    for dt in (torch.float32, torch.bfloat16):
                        D = torch.full((M, N), float("nan"), device=dev, dtype=dt)
                        mp.mp_gemm_ex(h, Ad, Bd, Cd, D, 1.25, beta, act=act)
                        torch.cuda.synchronize()
                        ok, worst = oracle.within_bound_out(D.float().cpu().numpy(), ref, mag, act,
                                                            dt == torch.bfloat16)
                        assert ok, (f"kernel {k} ({desc.um}x{desc.un} swap={desc.swap} pair={desc.pair}) "
                                    f"splits={splits} act={act} {dt} worst={worst:.3g}")
    finally:
        mp.mp_force_plan(h, -1, 0)


def test_activation_values_exact_inputs():
    """alpha = 0, beta = 1: D = act(C) with C exact, so the activation alone is
    measured, far below the GEMM bound: ReLU exactly; GELU within 1e-6 |x|
    (Hastings' erf approximation, 1.5e-7, plus fp32 rounding)."""
    import oracle
    dev = torch.device("cuda", 0)
    M, N, K = 256, 512, 64
    A, B, _ = rand_problem(M, N, K, seed=5, beta=0.0)
    x = np.linspace(-12.0, 12.0, M * N, dtype=np.float32).reshape(M, N)
    x[0, :8] = [0.0, -0.0, 1e-30, -1e-30, 3.0e4, -3.0e4, 0.5, -0.5]
    C = torch.from_numpy(x)
    h = handle()
    for act in (mp.MP_ACT_RELU, mp.MP_ACT_GELU):
        D = torch.empty(M, N, device=dev)
        mp.mp_gemm_ex(h, A.to(dev), B.to(dev), C.to(dev), D, 0.0, 1.0, act=act)
        torch.cuda.synchronize()
        got = D.cpu().numpy().astype(np.float64)
        ref = oracle.epilogue(x.astype(np.float64), act)
        if act == mp.MP_ACT_RELU:
            assert np.array_equal(got, ref)
        else:
            err = np.abs(got - ref)
            assert np.all(err <= 1e-6 * np.abs(x)), float((err / np.maximum(np.abs(x), 1e-30)).max())


def test_epilogue_word_zero_is_mp_gemm():
    """mp_gemm is mp_gemm_ex with epilogue 0: the same bits."""
    dev = torch.device("cuda", 0)
    for (M, N, K, beta) in [(1000, 768, 1300, 0.5), (105, 1024, 12544, 1.0), (4096, 4096, 512, 0.0)]:
        A, B, C = rand_problem(M, N, K, seed=K, beta=beta)
        Cd = C.to(dev) if C is not None else None
        D1 = torch.empty(M, N, device=dev)
        D2 = torch.empty(M, N, device=dev)
        mp.mp_gemm(handle(), A.to(dev), B.to(dev), Cd, D1, 1.0, beta)
        mp.mp_gemm_ex(handle(), A.to(dev), B.to(dev), Cd, D2, 1.0, beta, act=mp.MP_ACT_NONE)
        torch.cuda.synchronize()
        assert torch.equal(D1, D2)


def test_bounded_wait_reports_timeout_and_recovers():
    """A withheld pipeline stage makes the consumer's bounded wait expire; the
    kernel stops cleanly, mp_check reports it, and the next call is correct."""
    h = handle()
    dev = torch.device("cuda", 0)
    A, B, C = rand_problem(256, 256, 512, seed=2, beta=0.5)
    D = torch.empty(256, 256, device=dev)
    mp.mp_inject_wait_timeout(h, True, 50_000_000)  # 50 ms
    mp.mp_gemm(h, A.to(dev), B.to(dev), C.to(dev), D, 1.0, 0.5)
    assert mp.mp_check(h) == mp.MP_ERR_DEVICE_TIMEOUT
    mp.mp_inject_wait_timeout(h, False, 1_000_000_000)
    assert mp.mp_check(h) == mp.MP_OK
    D2 = run_gemm(A, B, C, 1.0, 0.5)
    assert_parity(D2, A, B, C, 1.0, 0.5, what="after timeout")


def test_bounded_waits_of_the_other_kernels_report_and_recover():
    """The same withheld stage in the fused pair, the convolution and the
    grouped GEMM: each kernel's bounded wait runs out, it stops cleanly,
    mp_check reports the timeout, and the next call is correct."""
    import oracle
    h = handle()
    dev = torch.device("cuda", 0)
    b = wl.B2B(256, 128, 256, 192, act0=1, seed=3)
    A0, W0, C0, W1, C1 = wl.make_b2b_operands(b)
    c = wl.Conv(2, 9, 9, 64, 64, seed=4)
    X, F, _ = wl.make_conv_operands(c)
    g = wl.Gemm(200, 300, 256, seed=5)
    A, B, _ = wl.make_operands(g)

    def fused():
        D1 = torch.empty(b.M, b.N1, device=dev)
        mp.mp_gemm_b2b(h, A0.to(dev), W0.to(dev), None, W1.to(dev), None, D1, 1.0, 0.0, 1.0, 0.0, b.act0)
        return D1

    def conv():
        D = torch.empty(c.N, c.P, c.Q, c.K, device=dev)
        mp.mp_conv2d(h, X.to(dev), F.to(dev), None, D)
        return D

    def grouped():
        D = torch.empty(g.M, g.N, device=dev)
        mp.mp_gemm_grouped(h, [(A.to(dev), B.to(dev), None, D, 1.0, 0.0)])
        return D

    mp.mp_set_b2b_mode(h, mp.MP_B2B_FUSED)
    try:
        for run in (fused, conv, grouped):
            mp.mp_inject_wait_timeout(h, True, 50_000_000)  # 50 ms
            run()
            assert mp.mp_check(h) == mp.MP_ERR_DEVICE_TIMEOUT, run.__name__
            mp.mp_inject_wait_timeout(h, False, 1_000_000_000)
            assert mp.mp_check(h) == mp.MP_OK
        bits = wl.bf16_bits
        D1 = fused().cpu().numpy()
        args = (bits(A0), bits(W0), None, bits(W1), None, 1.0, 0.0, 1.0, 0.0)
        ref, d0 = oracle.b2b(*args, b.act0)
        assert oracle.within_b2b(D1, ref, oracle.b2b_bound(*args, b.act0, d0))[0]
        D = conv().cpu().numpy().reshape(-1, c.K)
        assert oracle.within_bound(D, oracle.conv2d_nhwc(bits(X), bits(F)).reshape(-1, c.K),
                                   oracle.conv2d_magnitude(bits(X), bits(F)).reshape(-1, c.K))[0]
        D = grouped().cpu().numpy()
        assert oracle.within_bound(D, oracle.gemm(bits(A), bits(B)), oracle.magnitude(bits(A), bits(B)))[0]
    finally:
        mp.mp_set_b2b_mode(h, mp.MP_B2B_AUTO)
        mp.mp_inject_wait_timeout(h, False, 1_000_000_000)


# --------------------------------------------------------------------------
# split-K sums staged in the idle operand ring (a CTA's last unit)
# --------------------------------------------------------------------------
def _ring_kernels():
    ks = _kernels()
    normal = next(i for i, d in enumerate(ks) if not d.pair and not d.swap and d.un == 128)
    swapped = next(i for i, d in enumerate(ks) if d.swap and d.um == 32)
    return normal, swapped


@pytest.mark.parametrize("c_offset", [0, 1])
def test_ring_staged_split_sums(c_offset):
    """Twelve splits (more than a cluster holds on chip) of a few tiles: every
    CTA's only unit is a split, so its 1/S of the tile's rows are summed from
    partials bulk-copied into the idle ring.  Normal and swapped tiles, a
    ragged last row tile, beta * C with C's rows 16-byte aligned (copied into
    the ring too) and offset by 4 bytes (read directly), against the oracle."""
    h = handle()
    dev = torch.device("cuda", 0)
    normal, swapped = _ring_kernels()
    try:
        for k, (M, N, K) in [(normal, (200, 300, 2000)), (normal, (130, 256, 1500)),
                             (swapped, (50, 300, 2000)), (swapped, (77, 128, 1300))]:
            mp.mp_force_plan(h, k, 12)
            p = mp.mp_plan(h, M, N, K)
            assert p.total_tasks <= mp.mp_get_hw(h)[0].num_pe, "one unit per CTA"
            A, B, C = rand_problem(M, N, K, seed=M + K + c_offset, beta=0.5)
            # C stored with row pitch N + 4 starting c_offset floats into its buffer.
            store = torch.zeros(M * (N + 4) + 4, dtype=torch.float32, device=dev)
            Cv = store[c_offset:c_offset + M * (N + 4)].view(M, N + 4)[:, :N]
            Cv.copy_(C.to(dev))
            D = torch.full((M, N), float("nan"), device=dev)
            mp.mp_gemm(h, A.to(dev), B.to(dev), Cv, D, 1.5, 0.5)
            torch.cuda.synchronize()
            assert_parity(D.cpu(), A, B, C, 1.5, 0.5, what=f"ring sums kernel {k} {(M, N, K)} C+{4 * c_offset}B")
    finally:
        mp.mp_force_plan(h, -1, 0)


def test_ring_staged_split_sums_timeout_reports_and_recovers():
    """Hook mode 2: the ring-staged sums wait for 16 bytes more than are
    copied; the bounded wait runs out, mp_check reports it, and the next call
    is correct."""
    h = handle()
    dev = torch.device("cuda", 0)
    normal, _ = _ring_kernels()
    A, B, C = rand_problem(200, 300, 2000, seed=77, beta=0.5)
    try:
        mp.mp_force_plan(h, normal, 12)
        D = torch.empty(200, 300, device=dev)
        mp.mp_inject_wait_timeout(h, 2, 50_000_000)  # 50 ms
        mp.mp_gemm(h, A.to(dev), B.to(dev), C.to(dev), D, 1.0, 0.5)
        assert mp.mp_check(h) == mp.MP_ERR_DEVICE_TIMEOUT
        mp.mp_inject_wait_timeout(h, 0, 1_000_000_000)
        assert mp.mp_check(h) == mp.MP_OK
        assert_parity(run_gemm(A, B, C, 1.0, 0.5), A, B, C, 1.0, 0.5, what="after ring timeout")
    finally:
        mp.mp_inject_wait_timeout(h, 0, 1_000_000_000)
        mp.mp_force_plan(h, -1, 0)


@pytest.mark.parametrize("kernel_un", [64, 128, 192, 256])
def test_aligned_d_beta_c_every_width(kernel_un):
    """beta * C with 16-byte aligned rows of C and D (the bulk-store epilogue,
    C read a 32-column chunk at a time): one-wave and multi-wave plans,
    ragged last row tiles, tiles past N, in place and not, every normal tile
    width, against the oracle."""
    h = handle()
    dev = torch.device("cuda", 0)
    k = [i for i, d in enumerate(_kernels()) if (d.um, d.un, d.swap, d.pair) == (128, kernel_un, 0, 0)][0]
    try:
        mp.mp_force_plan(h, k, 1)
        for (M, N, K) in [(300, 1024, 200), (1000, 2048, 128), (37, 512, 64), (5000, 768, 96)]:
            A, B, C = rand_problem(M, N, K, seed=kernel_un + M, beta=0.5)
            D = run_gemm(A, B, C, 1.5, 0.5, h=h)
            assert_parity(D, A, B, C, 1.5, 0.5, what=f"aligned beta*C, 128x{kernel_un} {(M, N, K)}")
            CD = C.to(dev).clone()
            mp.mp_gemm(h, A.to(dev), B.to(dev), CD, CD, 1.5, 0.5)
            torch.cuda.synchronize()
            assert_parity(CD.cpu(), A, B, C, 1.5, 0.5, what=f"aligned beta*C in place, 128x{kernel_un} {(M, N, K)}")
    finally:
        mp.mp_force_plan(h, -1, 0)


# --------------------------------------------------------------------------
# the stress sweep: one GEMM of every plan class the polymerizer produces
# --------------------------------------------------------------------------
def _split_class(s):
    return "none" if s == 1 else ("on-chip-size" if s <= 8 else "wide")


def test_stress_every_plan_class():
    """The 1001 stress shapes (alpha 1.5, beta 0.5) fall into classes by
    (pattern, per region the micro-kernel and its split-K -- none, up to 8
    ways, more --, and whether A's, B's and D's rows are 16-byte aligned).
    The smallest shape of every class runs: the full oracle up to 2^30
    multiply-adds, else every entry of the edge tiles, 4096 random entries
    and a Freivalds probe of the whole product."""
    h = handle()
    gs = wl.workload("stress")
    classes = {}
    for g in gs:
        p = mp.mp_plan(h, g.M, g.N, g.K)
        key = (p.pattern, tuple((r.kernel, _split_class(r.splits)) for r in p.regions()),
               (2 * g.K) % 16 == 0, (2 * g.N) % 16 == 0, (4 * g.N) % 16 == 0)
        classes.setdefault(key, []).append(g)
    assert sum(len(v) for v in classes.values()) == len(gs) == 1001
    assert len(classes) >= 20, len(classes)
    rng = np.random.default_rng(11)
    for key in sorted(classes, key=str):
        g = min(classes[key], key=lambda x: x.flops)
        A, B, C = wl.make_operands(g)
        D = run_gemm(A, B, C, g.alpha, g.beta)
        what = f"stress class {key} via {(g.M, g.N, g.K)}"
        if g.M * g.N * g.K <= 2 ** 30:
            assert_parity(D, A, B, C, g.alpha, g.beta, what=what)
        else:
            assert_sampled_parity(D, A, B, C, g.alpha, g.beta, rng, what=what)

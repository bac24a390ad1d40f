"""Pins for the fp64 oracle, checked against what the pages and mathematics fix.

Each pin is written as a function of a GEMM callable so that the same checks
can be run against deliberately broken copies of the oracle (planted mistakes:
a dropped term, a wrong sign, a wrong index, a transposed operand, an
off-by-one loop) and shown to reject every one of them.
"""
import fractions
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from micro_polymerization_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_to_bf16_bits(x):
    """Round fp32 values to bf16 (nearest even) and return the bit patterns."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u >> 16) & 1) + 0x7FFF
    return ((u + r) >> 16).astype(np.uint16)


def rand_bits(rng, shape):
    return f32_to_bf16_bits(rng.uniform(-1, 1, size=shape).astype(np.float32))


def int_bits(rng, shape, lo=-4, hi=4):
    return f32_to_bf16_bits(rng.integers(lo, hi + 1, size=shape).astype(np.float32))


def exact_gemm(A, B, C, alpha, beta):
    """Exact rational D via fractions (independent of any float arithmetic)."""
    Af = [[fractions.Fraction(float(v)) for v in row] for row in oracle.bf16_bits_to_f64(A)]
    Bf = [[fractions.Fraction(float(v)) for v in row] for row in oracle.bf16_bits_to_f64(B)]
    M, K = A.shape
    N = B.shape[1]
    a, b = fractions.Fraction(alpha), fractions.Fraction(beta)
    D = [[None] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = sum((Af[i][k] * Bf[k][j] for k in range(K)), fractions.Fraction(0))
            c = fractions.Fraction(float(C[i, j])) if beta != 0 else 0
            D[i][j] = a * s + b * c
    return D


# ----------------------------------------------------------------------------
# Pins (each takes a callable gemm(A_bits, B_bits, C, alpha, beta) -> fp64 D)
# ----------------------------------------------------------------------------

def pin_widening():
    table = {0x3F80: 1.0, 0xC000: -2.0, 0x0000: 0.0, 0x8000: -0.0, 0x3F00: 0.5,
             0x0001: 2.0 ** -133, 0x7F7F: (2 - 2 ** -7) * 2.0 ** 127, 0x4049: 3.140625}
    got = oracle.bf16_bits_to_f64(np.array(list(table), dtype=np.uint16))
    return np.array_equal(got, np.array(list(table.values())))


def pin_closed_form_ones(gemm):
    """A = 1, B = 1:  D = alpha*K + beta*C  exactly (ragged and odd sizes)."""
    rng = np.random.default_rng(5)
    for (M, N, K) in [(3, 5, 7), (33, 17, 65), (1, 1, 1), (2, 70, 129)]:
        A = np.full((M, K), 0x3F80, dtype=np.uint16)
        B = np.full((K, N), 0x3F80, dtype=np.uint16)
        C = rng.integers(-8, 9, size=(M, N)).astype(np.float32)
        for alpha, beta in [(1.0, 0.0), (1.5, 0.5), (-2.0, 1.0), (0.25, -3.0)]:
            D = gemm(A, B, C, alpha, beta)
            want = alpha * K + beta * C.astype(np.float64)
            if not np.array_equal(D, want):
                return False
    return True


def pin_identity_permutation(gemm):
    """B = I gives alpha*A + beta*C; B = P (a permutation) permutes A's columns."""
    rng = np.random.default_rng(6)
    M, K = 9, 13
    A = rand_bits(rng, (M, K))
    Af = oracle.bf16_bits_to_f64(A)
    C = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    eye = np.where(np.eye(K, dtype=bool), 0x3F80, 0).astype(np.uint16)
    D = gemm(A, eye, C, 1.0, 0.5)
    if not np.array_equal(D, Af + 0.5 * C.astype(np.float64)):
        return False
    perm = rng.permutation(K)
    P = np.zeros((K, K), dtype=np.uint16)
    P[perm, np.arange(K)] = 0x3F80  # column j of P selects row perm[j] of ... A[:, perm[j]]
    D = gemm(A, P, C, 1.0, 0.0)
    return np.array_equal(D, Af[:, perm])


def pin_bruteforce_exact(gemm):
    """Tiny non-square shapes vs the exact rational result, within fp64 rounding."""
    rng = np.random.default_rng(7)
    for (M, N, K) in [(1, 1, 1), (2, 3, 4), (4, 3, 2), (5, 1, 3), (3, 4, 5), (6, 2, 7)]:
        A = rand_bits(rng, (M, K))
        B = rand_bits(rng, (K, N))
        C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
        for alpha, beta in [(1.0, 0.0), (1.5, 0.5), (-0.75, 2.0)]:
            D = gemm(A, B, C, alpha, beta)
            E = exact_gemm(A, B, C, alpha, beta)
            mag = (abs(alpha) * (np.abs(oracle.bf16_bits_to_f64(A)) @ np.abs(oracle.bf16_bits_to_f64(B)))
                   + abs(beta) * np.abs(C.astype(np.float64)))
            for i in range(M):
                for j in range(N):
                    err = abs(fractions.Fraction(float(D[i, j])) - E[i][j])
                    if err > fractions.Fraction((K + 4) * 2.0 ** -52 * mag[i, j]):
                        return False
    return True


def pin_integer_exact(gemm):
    """Integer-valued operands: every partial sum is exact, so D is exact."""
    rng = np.random.default_rng(8)
    for (M, N, K) in [(64, 96, 32), (37, 45, 70), (1, 33, 65)]:
        A = int_bits(rng, (M, K))
        B = int_bits(rng, (K, N))
        C = rng.integers(-4, 5, size=(M, N)).astype(np.float32)
        want = (oracle.bf16_bits_to_f64(A).astype(np.int64) @ oracle.bf16_bits_to_f64(B).astype(np.int64)
                ).astype(np.float64) * 2.0 + 3.0 * C
        if not np.array_equal(gemm(A, B, C, 2.0, 3.0), want):
            return False
    return True


def pin_fp64_cancellation(gemm):
    """1 + 2^-30 - 1 = 2^-30 holds in fp64 (the oracle's precision) but not in
    fp32: the accumulation must be carried in fp64."""
    A = np.array([[0x3F80, 0x3080, 0xBF80]], dtype=np.uint16)  # 1, 2^-30, -1
    B = np.full((3, 2), 0x3F80, dtype=np.uint16)
    D = gemm(A, B, None, 1.0, 0.0)
    return np.array_equal(D, np.full((1, 2), 2.0 ** -30))


ORACLE_FORMS = {
    "naive": lambda A, B, C, a, b: oracle.gemm_naive(A, B, C, a, b),
    "tiled": lambda A, B, C, a, b: oracle.gemm_tiled(A, B, C, a, b),
    "rows": lambda A, B, C, a, b: oracle.gemm(A, B, C, a, b),
}


def _entries_form(A, B, C, a, b):
    M, N = A.shape[0], B.shape[1]
    r, c = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    out, _ = oracle.gemm_entries(A, B, C, a, b, r.ravel(), c.ravel())
    return out.reshape(M, N)


ORACLE_FORMS["entries"] = _entries_form
PINS = [pin_closed_form_ones, pin_identity_permutation, pin_bruteforce_exact, pin_integer_exact,
        pin_fp64_cancellation]


def test_bf16_widening():
    assert pin_widening()


@pytest.mark.parametrize("form", sorted(ORACLE_FORMS))
@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pins(form, pin):
    assert pin(ORACLE_FORMS[form])


@pytest.mark.parametrize("M,N,K", [(64, 64, 64), (96, 32, 128), (37, 45, 70), (33, 1, 31), (1, 65, 97)])
def test_naive_equals_tiled_bitwise(M, N, K):
    """The two printed nests (MikPoly summary, preliminaries part 2) agree exactly on
    integer data, for tile-multiple and ragged sizes."""
    rng = np.random.default_rng(M * 1000 + N * 10 + K)
    A, B = int_bits(rng, (M, K)), int_bits(rng, (K, N))
    C = rng.integers(-4, 5, size=(M, N)).astype(np.float32)
    Dn = oracle.gemm_naive(A, B, C, 1.0, 1.0)
    Dt = oracle.gemm_tiled(A, B, C, 1.0, 1.0)
    Dr = oracle.gemm(A, B, C, 1.0, 1.0)
    assert np.array_equal(Dn, Dt) and np.array_equal(Dn, Dr)


def test_forms_agree_on_random_data():
    """Same k order in every form: naive, rows and entries are bitwise equal;
    the tiled nest sums the same terms in the same order as well."""
    rng = np.random.default_rng(11)
    A, B = rand_bits(rng, (21, 40)), rand_bits(rng, (40, 19))
    C = rng.uniform(-1, 1, size=(21, 19)).astype(np.float32)
    ref = oracle.gemm_naive(A, B, C, 1.5, 0.5)
    for name, f in ORACLE_FORMS.items():
        assert np.array_equal(f(A, B, C, 1.5, 0.5), ref), name


def test_beta_zero_never_reads_c():
    rng = np.random.default_rng(12)
    A, B = rand_bits(rng, (4, 5)), rand_bits(rng, (5, 6))
    C = np.full((4, 6), np.nan, dtype=np.float32)
    for f in ORACLE_FORMS.values():
        assert np.all(np.isfinite(f(A, B, C, 1.0, 0.0)))


def test_k_zero_gives_beta_c():
    rng = np.random.default_rng(13)
    A = np.zeros((3, 0), dtype=np.uint16)
    B = np.zeros((0, 4), dtype=np.uint16)
    C = rng.uniform(-1, 1, size=(3, 4)).astype(np.float32)
    for f in ORACLE_FORMS.values():
        assert np.array_equal(f(A, B, C, 2.0, 0.5), 0.5 * C.astype(np.float64))


def test_leading_dimensions():
    """Padded leading dimensions address the same logical matrices."""
    rng = np.random.default_rng(14)
    A, B = rand_bits(rng, (7, 9)), rand_bits(rng, (9, 5))
    C = rng.uniform(-1, 1, size=(7, 5)).astype(np.float32)
    Ap = np.zeros((7, 16), np.uint16); Ap[:, :9] = A
    Bp = np.zeros((9, 11), np.uint16); Bp[:, :5] = B
    Cp = np.zeros((7, 8), np.float32); Cp[:, :5] = C
    ref = oracle.gemm_naive(A, B, C, 1.0, 1.0)
    for f in ORACLE_FORMS.values():
        assert np.array_equal(f(Ap[:, :9], Bp[:, :5], Cp[:, :5], 1.0, 1.0), ref)


def test_magnitude_closed_form():
    A = np.full((3, 10), 0xBF80, dtype=np.uint16)  # -1
    B = np.full((10, 4), 0x4000, dtype=np.uint16)  # 2
    C = np.full((3, 4), -3.0, dtype=np.float32)
    G = oracle.magnitude(A, B, C, beta=0.5)
    assert np.array_equal(G, np.full((3, 4), 20.0 + 1.5))


def test_freivalds_separates_right_from_wrong():
    rng = np.random.default_rng(15)
    M, N, K = 40, 30, 50
    A, B = rand_bits(rng, (M, K)), rand_bits(rng, (K, N))
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    D = oracle.gemm(A, B, C, 1.5, 0.5).astype(np.float32)
    x = rng.choice([-1.0, 1.0], size=N)
    y, ymag = oracle.freivalds(A, B, C, 1.5, 0.5, D, x)
    assert np.all(np.abs(y) <= 1e-5 * ymag + 1e-12)
    D2 = D.copy()
    D2[17, 3] += 0.05
    y, ymag = oracle.freivalds(A, B, C, 1.5, 0.5, D2, x)
    assert np.abs(y[17]) > 1e-5 * ymag[17] and np.all(np.abs(np.delete(y, 17)) <= 1e-5 * np.delete(ymag, 17))


def test_within_bound_semantics():
    ok, r = oracle.within_bound(np.array([1.0, 2.0]), np.array([1.0, 2.001]), np.array([1.0, 1.0]))
    assert ok and 0.4 < r < 0.6
    ok, _ = oracle.within_bound(np.array([1.0]), np.array([1.003]), np.array([1.0]))
    assert not ok
    ok, _ = oracle.within_bound(np.array([np.nan]), np.array([0.0]), np.array([1.0]))
    assert not ok
    ok, _ = oracle.within_bound(np.array([0.0]), np.array([1e-30]), np.array([0.0]))
    assert not ok


# ----------------------------------------------------------------------------
# Planted mistakes: broken copies of the definition (numpy, fp64) must each
# fail at least one pin.  The mistakes live here, on the CPU, never in the
# oracle's sources.
# ----------------------------------------------------------------------------

def _f(bits):
    return oracle.bf16_bits_to_f64(bits)


def _c(C, beta, shape):
    return beta * C.astype(np.float64) if beta != 0 else np.zeros(shape)


MUTANTS = {
    "dropped_beta_term": lambda A, B, C, a, b: a * (_f(A) @ _f(B)),
    "wrong_beta_sign": lambda A, B, C, a, b: a * (_f(A) @ _f(B)) - _c(C, b, (A.shape[0], B.shape[1])),
    "alpha_on_c": lambda A, B, C, a, b: a * (_f(A) @ _f(B) + _c(C, b, (A.shape[0], B.shape[1]))),
    "k_off_by_one": lambda A, B, C, a, b: a * (_f(A)[:, :-1] @ _f(B)[:-1, :]) + _c(C, b, (A.shape[0], B.shape[1])),
    "b_transposed": lambda A, B, C, a, b: (a * (_f(A) @ _f(B).T.reshape(B.shape))
                                            + _c(C, b, (A.shape[0], B.shape[1]))),
    "a_rows_reversed": lambda A, B, C, a, b: a * (_f(A)[::-1] @ _f(B)) + _c(C, b, (A.shape[0], B.shape[1])),
    "products_in_fp32": lambda A, B, C, a, b: (a * (_f(A).astype(np.float32) @ _f(B).astype(np.float32))
                                                .astype(np.float64) + _c(C, b, (A.shape[0], B.shape[1]))),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistakes(name):
    mutant = MUTANTS[name]

    def safe(pin):
        try:
            return pin(mutant)
        except Exception:
            return False

    assert not all(safe(p) for p in PINS), f"no pin caught {name}"


def test_correct_numpy_restatement_passes_pins():
    """Control for the planted-mistake test: an independent fp64 numpy
    statement of the definition passes the same pins."""
    good = lambda A, B, C, a, b: a * (_f(A) @ _f(B)) + _c(C, b, (A.shape[0], B.shape[1]))
    assert pin_closed_form_ones(good) and pin_identity_permutation(good) and pin_integer_exact(good)


# ----------------------------------------------------------------------------
# Workload recipe sanity (shared generator module; no arithmetic of the method)
# ----------------------------------------------------------------------------

def test_workload_shapes_follow_their_recipes():
    seq = wl.dynamic_sequence()
    assert len(seq) == 64 and all(g.M % 8 == 0 and 8 <= g.M <= 4096 for g in seq)
    assert [(g.N, g.K) for g in seq[:4]] == wl.SEQ_NK
    conv = wl.dynamic_resolution()
    assert all(g.N in (64, 128, 256, 512) and g.K == 9 * g.N for g in conv)
    qkv = wl.merged_qkv()
    assert all(g.N == 3072 and g.K == 1024 and 1 <= g.M <= 4096 for g in qkv)
    bat = wl.merged_batched()
    assert all(g.batch == 12 and g.K == 64 and g.M == g.N and 16 <= g.M <= 512 for g in bat)
    st = wl.stress()
    assert len(st) == 1001 and st[-1].M == st[-1].N == st[-1].K == 4096
    assert all(1 <= d <= 16384 for g in st for d in (g.M, g.N, g.K))
    assert wl.single_skinny()[0].M == 105


def test_generator_is_seeded_and_in_range():
    g = wl.Gemm(17, 9, 33, alpha=1.5, beta=0.5, seed=42)
    A1, B1, C1 = wl.make_operands(g)
    A2, B2, C2 = wl.make_operands(g)
    assert np.array_equal(wl.bf16_bits(A1), wl.bf16_bits(A2))
    assert np.array_equal(C1.numpy(), C2.numpy())
    for T in (A1.float(), B1.float(), C1):
        assert float(T.min()) >= -1.0 and float(T.max()) <= 1.0
    # torch's bf16 rounding agrees with round-to-nearest-even of the fp32 draw
    x = np.random.default_rng(0).uniform(-1, 1, 1000).astype(np.float32)
    import torch
    assert np.array_equal(wl.bf16_bits(torch.from_numpy(x).to(torch.bfloat16)), f32_to_bf16_bits(x))


# ----------------------------------------------------------------------------
# Epilogue variants: activations and bf16 output
# ----------------------------------------------------------------------------

def test_activation_pins():
    """ReLU's closed form; GELU = x*Phi(x) against standard-normal table values
    (Phi(1) = 0.8413447460685429, Phi(-1) = 0.15865525393145707,
    Phi(2) = 0.9772498680518208), the identity gelu(x) - gelu(-x) = x, and its
    tails."""
    x = np.array([-3.0, -1.0, -0.0, 0.0, 0.5, 1.0, 2.0, 40.0])
    assert np.array_equal(oracle.epilogue(x, oracle.ACT_RELU), np.maximum(x, 0.0))
    assert np.array_equal(oracle.epilogue(x, oracle.ACT_NONE), x)
    g = oracle.epilogue(np.array([1.0, -1.0, 2.0]), oracle.ACT_GELU)
    assert np.allclose(g, [0.8413447460685429, -0.15865525393145707, 2 * 0.9772498680518208], rtol=0, atol=1e-15)
    y = np.linspace(-6, 6, 241)
    assert np.allclose(oracle.epilogue(y, oracle.ACT_GELU) - oracle.epilogue(-y, oracle.ACT_GELU), y, atol=1e-14)
    assert abs(oracle.epilogue(np.array([40.0]), oracle.ACT_GELU)[0] - 40.0) < 1e-12
    assert abs(oracle.epilogue(np.array([-40.0]), oracle.ACT_GELU)[0]) < 1e-12
    # the slope bound used by the parity check
    h = 1e-6
    slope = (oracle.epilogue(y + h, oracle.ACT_GELU) - oracle.epilogue(y - h, oracle.ACT_GELU)) / (2 * h)
    assert slope.max() <= oracle.ACT_SLOPE[oracle.ACT_GELU] and slope.max() > 1.12


def test_bf16_rounding_pins():
    """Nearest-even rounding to bf16: exact values stay, halfway cases go to
    the even neighbour, and the result matches torch's own conversion."""
    import torch
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 3.0e38, 1e-40])
    r = oracle.bf16_round(vals)
    assert r[0] == 1.0 and r[1] == 1.0 and r[2] == 1.0 + 4 * 2 ** -8 and r[3] == 1.0 and r[4] == -2.5
    rng = np.random.default_rng(3)
    x = rng.standard_normal(10000) * 10.0 ** rng.integers(-6, 6, 10000)
    t = torch.tensor(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.bf16_round(x.astype(np.float32).astype(np.float64)), t)


# ---------------------------------------------------------------------------
# Back-to-back GEMMs (BOLT summary, persistent kernel (GEMM/Conv) fusion)
# ---------------------------------------------------------------------------
def oracle_bits(rng, shape):
    """uniform[-1, 1) values cut to bf16 bit patterns (any bf16 values serve)."""
    v = rng.uniform(-1, 1, size=shape).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


def _int_bf16(rng, shape, lo=-3, hi=4):
    """Small integers: exact in bf16, and every sum below stays exact in fp64."""
    v = rng.integers(lo, hi, size=shape).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16), v.astype(np.float64)


def test_b2b_brute_force_small():
    """Pure-Python loops over the two formulas on tiny integer inputs: exact
    for no activation and ReLU, within 1e-12 for GELU."""
    import math
    rng = np.random.default_rng(7)
    M, K0, N0, N1 = 3, 5, 4, 2
    A0, a0 = _int_bf16(rng, (M, K0))
    W0, w0 = _int_bf16(rng, (K0, N0))
    W1, w1 = _int_bf16(rng, (N0, N1))
    C0 = rng.integers(-5, 6, size=(M, N0)).astype(np.float32)
    C1 = rng.integers(-5, 6, size=(M, N1)).astype(np.float32)
    al0, be0, al1, be1 = 2.0, -1.0, 0.5, 3.0

    def act(x, a):
        if a == oracle.ACT_RELU:
            return max(x, 0.0)
        if a == oracle.ACT_GELU:
            return x * 0.5 * (1.0 + math.erf(x / math.sqrt(2.0)))
        return x

    for a in (oracle.ACT_NONE, oracle.ACT_RELU, oracle.ACT_GELU):
        ref = np.zeros((M, N1))
        for r in range(M):
            d0 = []
            for k in range(N0):
                s = 0.0
                for i in range(K0):
                    s += a0[r, i] * w0[i, k]
                d0.append(act(al0 * s + be0 * float(C0[r, k]), a))
            for j in range(N1):
                t = 0.0
                for k in range(N0):
                    t += d0[k] * w1[k, j]
                ref[r, j] = al1 * t + be1 * float(C1[r, j])
        D1, _ = oracle.b2b(A0, W0, C0, W1, C1, al0, be0, al1, be1, a)
        if a == oracle.ACT_GELU:
            assert np.allclose(D1, ref, rtol=0, atol=1e-12)
        else:
            assert np.array_equal(D1, ref)


def test_b2b_associativity():
    """No activation and beta0 = 0: D1 = alpha1 alpha0 A0 (W0 W1) + beta1 C1,
    the product taken in the other order, exact on integer inputs; a transposed
    or swapped operand fails it."""
    rng = np.random.default_rng(11)
    M, K0, N0, N1 = 9, 7, 6, 5
    A0, a0 = _int_bf16(rng, (M, K0))
    W0, w0 = _int_bf16(rng, (K0, N0))
    W1, w1 = _int_bf16(rng, (N0, N1))
    C1 = rng.integers(-5, 6, size=(M, N1)).astype(np.float32)
    D1, _ = oracle.b2b(A0, W0, None, W1, C1, 3.0, 0.0, -2.0, 0.5)
    assert np.array_equal(D1, -6.0 * (a0 @ (w0 @ w1)) + 0.5 * C1)


def test_b2b_identity_second_gemm_is_epilogue_gemm():
    """W1 = I, alpha1 = 1, beta1 = 0: D1 is the first GEMM with its activation."""
    rng = np.random.default_rng(3)
    M, K0, N0 = 17, 40, 24
    A0 = oracle_bits(rng, (M, K0))
    W0 = oracle_bits(rng, (K0, N0))
    C0 = rng.uniform(-1, 1, size=(M, N0)).astype(np.float32)
    eye = (np.eye(N0, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    for a in (oracle.ACT_NONE, oracle.ACT_RELU, oracle.ACT_GELU):
        D1, D0 = oracle.b2b(A0, W0, C0, eye, None, 1.5, 0.25, 1.0, 0.0, a)
        assert np.array_equal(D1, oracle.epilogue(oracle.gemm(A0, W0, C0, 1.5, 0.25), a))
        assert np.array_equal(D1, D0)


def _fp32_b2b(A0, W0, C0, W1, C1, al0, be0, al1, be1, a, drop=None):
    """The fused kernel's precision path in numpy: fp32 products, D0 rounded to
    bf16 on chip.  `drop` plants one mistake."""
    f = lambda b: oracle.bf16_bits_to_f64(b).astype(np.float32)
    d0 = np.float32(al0) * (f(A0) @ f(W0))
    if be0 != 0.0 and drop != "beta0":
        d0 = d0 + np.float32(be0) * C0
    if drop != "act":
        d0 = oracle.epilogue(d0.astype(np.float64), a).astype(np.float32)
    d0 = oracle.bf16_round(d0).astype(np.float32)
    w1 = f(W1).T if drop == "transpose" else f(W1)
    d1 = np.float32(al1) * (d0 @ w1)
    if be1 != 0.0 and drop != "beta1":
        d1 = d1 + np.float32(be1) * C1
    return d1.astype(np.float64)


def test_b2b_bound_admits_fused_precision_and_rejects_mistakes():
    rng = np.random.default_rng(5)
    M, K0, N0, N1 = 64, 96, 80, 80
    A0 = oracle_bits(rng, (M, K0))
    W0 = oracle_bits(rng, (K0, N0))
    W1 = oracle_bits(rng, (N0, N1))
    C0 = rng.uniform(-1, 1, size=(M, N0)).astype(np.float32)
    C1 = rng.uniform(-1, 1, size=(M, N1)).astype(np.float32)
    args = (A0, W0, C0, W1, C1, 1.25, 0.75, 0.5, 1.5)
    for a in (oracle.ACT_NONE, oracle.ACT_RELU, oracle.ACT_GELU):
        ref, d0 = oracle.b2b(*args, a)
        bound = oracle.b2b_bound(*args, a, d0)
        ok, worst = oracle.within_b2b(_fp32_b2b(*args, a), ref, bound)
        assert ok, worst
        for mistake in ("beta0", "beta1", "transpose") + (("act",) if a != oracle.ACT_NONE else ()):
            ok, worst = oracle.within_b2b(_fp32_b2b(*args, a, drop=mistake), ref, bound)
            assert not ok, (a, mistake, worst)


# ---------------------------------------------------------------------------
# Convolution (MikPoly summary, section 5: convolutions run as GEMM)
# ---------------------------------------------------------------------------
def _int_bits(rng, shape, lo=-3, hi=4):
    v = rng.integers(lo, hi, size=shape).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16), v.astype(np.float64)


def test_conv_brute_force_small():
    """Seven nested Python loops over the definition, integer inputs: exact."""
    rng = np.random.default_rng(21)
    for (N, H, W, C, K, R, S, ph, pw) in [(2, 4, 3, 3, 2, 3, 3, 1, 1), (1, 5, 5, 2, 3, 3, 3, 0, 0),
                                         (1, 3, 6, 2, 2, 1, 3, 0, 2), (2, 2, 2, 1, 1, 3, 3, 2, 1)]:
        X, x = _int_bits(rng, (N, H, W, C))
        Wt, w = _int_bits(rng, (R, S, C, K))
        Cin_shape = (N, H + 2 * ph - R + 1, W + 2 * pw - S + 1, K)
        Cin = rng.integers(-5, 6, size=Cin_shape).astype(np.float32)
        P, Q = Cin_shape[1], Cin_shape[2]
        ref = np.zeros(Cin_shape)
        for n in range(N):
            for p in range(P):
                for q in range(Q):
                    for k in range(K):
                        acc = 0.0
                        for r in range(R):
                            for s in range(S):
                                h, ww = p + r - ph, q + s - pw
                                if 0 <= h < H and 0 <= ww < W:
                                    for c in range(C):
                                        acc += x[n, h, ww, c] * w[r, s, c, k]
                        ref[n, p, q, k] = 2.0 * acc - 0.5 * Cin[n, p, q, k]
        D = oracle.conv2d_nhwc(X, Wt, Cin, 2.0, -0.5, ph, pw)
        assert np.array_equal(D, ref), (N, H, W, C, K, R, S, ph, pw)


def test_conv_is_gemm_on_im2col():
    """A GEMM-based convolution: the C GEMM oracle on the explicit im2col
    matrix and the filter as [R*S*C, K] gives the same values."""
    rng = np.random.default_rng(22)
    N, H, W, C, K = 2, 7, 9, 16, 24
    X = oracle_bits(rng, (N, H, W, C))
    Wt = oracle_bits(rng, (3, 3, C, K))
    Cin = rng.uniform(-1, 1, size=(N, H, W, K)).astype(np.float32)
    D = oracle.conv2d_nhwc(X, Wt, Cin, 1.5, 0.25)
    A = oracle.im2col_nhwc(X, 3, 3)
    G = oracle.gemm(A, Wt.reshape(9 * C, K), Cin.reshape(N * H * W, K), 1.5, 0.25)
    assert np.allclose(D.reshape(N * H * W, K), G, rtol=1e-12, atol=1e-12)
    mag = oracle.conv2d_magnitude(X, Wt, Cin, 0.25).reshape(N * H * W, K)
    assert np.allclose(mag, oracle.magnitude(A, Wt.reshape(9 * C, K), Cin.reshape(N * H * W, K), 0.25), rtol=1e-12)


def test_conv_1x1_is_gemm_and_delta_filter_is_identity():
    rng = np.random.default_rng(23)
    N, H, W, C, K = 3, 5, 4, 8, 6
    X = oracle_bits(rng, (N, H, W, C))
    Wt = oracle_bits(rng, (1, 1, C, K))
    D = oracle.conv2d_nhwc(X, Wt, pad_h=0, pad_w=0)
    assert np.array_equal(D.reshape(N * H * W, K), oracle.gemm(X.reshape(N * H * W, C), Wt.reshape(C, K)))
    # Centre tap = identity (C = K): a 3x3 "same" convolution returns its input.
    delta = np.zeros((3, 3, C, C), dtype=np.float32)
    delta[1, 1] = np.eye(C)
    db = (delta.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(oracle.conv2d_nhwc(X, db), oracle.bf16_bits_to_f64(X))


def test_conv_ones_closed_form():
    """All-ones input and filter, padding 1: each output counts its valid taps,
    C * rows(p) * cols(q), with rows(p) = 3 minus the taps off the top or
    bottom edge (likewise for columns)."""
    N, H, W, C, K = 1, 6, 5, 4, 2
    one = np.uint16(0x3F80)
    X = np.full((N, H, W, C), one, dtype=np.uint16)
    Wt = np.full((3, 3, C, K), one, dtype=np.uint16)
    D = oracle.conv2d_nhwc(X, Wt)
    valid = lambda i, n: 3 - (i == 0) - (i == n - 1)
    for p in range(H):
        for q in range(W):
            assert np.all(D[0, p, q] == C * valid(p, H) * valid(q, W))


def test_gemm_group_is_each_problem_and_matches_batched_case():
    """A group of same-shape problems is the batched GEMM (the merge of the
    BladeDISC notes): stacked, the group's results equal one fp64 product per
    problem computed with numpy on the widened values."""
    rng = np.random.default_rng(31)
    probs = []
    for i in range(5):
        A = oracle_bits(rng, (7, 11))
        B = oracle_bits(rng, (11, 6))
        C = rng.uniform(-1, 1, size=(7, 6)).astype(np.float32)
        probs.append((A, B, C, 1.0 + i, 0.5))
    out = oracle.gemm_group(probs)
    for (A, B, C, al, be), (D, mag) in zip(probs, out):
        ref = al * (oracle.bf16_bits_to_f64(A) @ oracle.bf16_bits_to_f64(B)) + be * C.astype(np.float64)
        assert np.allclose(D, ref, rtol=1e-13, atol=1e-13)
        assert np.all(mag >= np.abs(D - be * C) / al - 1e-12)
    # Different shapes in one group: each keeps its own shape.
    shapes = [(3, 5, 2), (1, 64, 9), (17, 3, 33)]
    probs = [(oracle_bits(rng, (m, k)), oracle_bits(rng, (k, n)), None, 1.0, 0.0) for m, n, k in shapes]
    assert [d.shape for d, _ in oracle.gemm_group(probs)] == [(m, n) for m, n, _ in shapes]

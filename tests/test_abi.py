"""The C-ABI library loads, exports every symbol include/mp.h declares, and
rejects bad arguments with status codes (no GPU needed: a planning-only
handle checks arguments before it would launch)."""
import ctypes
import os
import re

import numpy as np
import pytest

import micro_polymerization_gb300 as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^\s*(?:mp_status|const char\*)\s+(mp_\w+)\s*\(", text, re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("mp_init", "mp_destroy", "mp_plan", "mp_gemm", "mp_gemm_batched", "mp_status_string"):
        assert required in names


@pytest.mark.parametrize("name", declared_functions())
def test_library_exports_every_declared_symbol(name):
    lib = mp.library()
    assert hasattr(lib, name), name


def test_status_strings():
    for code in range(0, -7, -1):
        s = mp.mp_status_string(code)
        assert s and s != "unknown status"
    assert mp.mp_status_string(-99) == "unknown status"


def _host():
    hw = mp.MpHw(num_pe=148, warps_per_wave=888, local_mem_bytes=232448, shared_mem_bytes=1 << 27,
                 hbm_gbs=6684.0, l2_gbs=20000.0, mma_tflops=1974.0)
    return mp.mp_init_host(hw)


def test_argument_checks_before_launch():
    lib = mp.library()
    h = _host()
    A, B, C, D = 0x10000, 0x20000000, 0x30000000, 0x40000000  # never dereferenced
    g = lambda *a: lib.mp_gemm(h.ptr, *a)
    # valid request on a planning-only handle: unsupported, not invalid
    assert g(64, 64, 64, A, 64, B, 64, C, 64, D, 64, 1.0, 1.0, None) == mp.MP_ERR_UNSUPPORTED
    assert g(-1, 64, 64, A, 64, B, 64, C, 64, D, 64, 1.0, 0.0, None) == mp.MP_ERR_INVALID_ARG
    assert g(64, 64, 64, A, 63, B, 64, C, 64, D, 64, 1.0, 0.0, None) == mp.MP_ERR_INVALID_ARG  # lda < K
    assert g(64, 64, 64, A, 64, B, 63, C, 64, D, 64, 1.0, 0.0, None) == mp.MP_ERR_INVALID_ARG  # ldb < N
    assert g(64, 64, 64, A, 64, B, 64, C, 64, D, 63, 1.0, 0.0, None) == mp.MP_ERR_INVALID_ARG  # ldd < N
    assert g(64, 64, 64, A, 64, B, 64, None, 64, D, 64, 1.0, 0.5, None) == mp.MP_ERR_INVALID_ARG  # beta, no C
    assert g(64, 64, 64, None, 64, B, 64, None, 0, D, 64, 1.0, 0.0, None) == mp.MP_ERR_INVALID_ARG
    assert g(64, 64, 64, A, 64, B, 64, None, 0, None, 64, 1.0, 0.0, None) == mp.MP_ERR_INVALID_ARG
    assert g(64, 64, 64, A + 1, 64, B, 64, None, 0, D, 64, 1.0, 0.0, None) == mp.MP_ERR_INVALID_ARG  # odd bf16
    assert g(64, 64, 64, A, 64, B, 64, None, 0, D + 2, 64, 1.0, 0.0, None) == mp.MP_ERR_INVALID_ARG  # fp32 align
    # D overlapping A
    assert g(64, 64, 64, A, 64, B, 64, None, 0, A + 64, 64, 1.0, 0.0, None) == mp.MP_ERR_INVALID_ARG
    # D == C in place is fine (only with ldc == ldd)
    assert g(64, 64, 64, A, 64, B, 64, D, 64, D, 64, 1.0, 1.0, None) == mp.MP_ERR_UNSUPPORTED
    assert g(64, 64, 64, A, 64, B, 64, D, 80, D, 64, 1.0, 1.0, None) == mp.MP_ERR_INVALID_ARG
    # beta == 0 never needs C; empty problems are no-ops even here
    assert g(0, 64, 64, A, 64, B, 64, None, 0, D, 64, 1.0, 0.0, None) == mp.MP_OK
    assert g(64, 0, 64, A, 64, B, 1, None, 0, D, 1, 1.0, 0.0, None) == mp.MP_OK
    # batched: overlapping D blocks are rejected
    gb = lambda *a: lib.mp_gemm_batched(h.ptr, *a)
    assert gb(3, 8, 8, 8, A, 8, 64, B, 8, 64, None, 0, 0, D, 8, 32, 1.0, 0.0, None) == mp.MP_ERR_INVALID_ARG
    assert gb(3, 8, 8, 8, A, 8, 64, B, 8, 64, None, 0, 0, D, 8, 64, 1.0, 0.0, None) == mp.MP_ERR_UNSUPPORTED
    assert gb(3, 8, 8, 8, A, 8, -1, B, 8, 64, None, 0, 0, D, 8, 64, 1.0, 0.0, None) == mp.MP_ERR_INVALID_ARG
    h.close()


def test_plan_search_entry_points_check_arguments():
    """mp_enumerate_plans, mp_gemm_with_plan and mp_set_plan_mode reject bad
    arguments with status codes; a planning-only handle plans but cannot run."""
    lib = mp.library()
    h = _host()
    n = ctypes.c_int32(-1)
    e = lambda *a: lib.mp_enumerate_plans(*a)
    assert e(None, 1, 10, 10, 10, None, 0, ctypes.byref(n)) == mp.MP_ERR_INVALID_ARG
    assert e(h.ptr, 1, 10, 10, 10, None, -1, ctypes.byref(n)) == mp.MP_ERR_INVALID_ARG
    assert e(h.ptr, 1, 10, 10, 10, None, 5, ctypes.byref(n)) == mp.MP_ERR_INVALID_ARG  # capacity without array
    assert e(h.ptr, 1, 0, 10, 10, None, 0, ctypes.byref(n)) == mp.MP_ERR_INVALID_ARG
    assert e(h.ptr, 1, 10, 10, 10, None, 0, None) == mp.MP_ERR_INVALID_ARG
    assert e(h.ptr, 1, 100, 100, 100, None, 0, ctypes.byref(n)) == mp.MP_OK and n.value > 0
    assert lib.mp_set_plan_mode(None, 0) == mp.MP_ERR_INVALID_ARG
    assert lib.mp_set_plan_mode(h.ptr, 3) == mp.MP_ERR_INVALID_ARG
    assert lib.mp_set_plan_mode(h.ptr, mp.MP_PLAN_WAVE) == mp.MP_OK
    assert lib.mp_set_plan_mode(h.ptr, mp.MP_PLAN_MIKPOLY) == mp.MP_OK
    plan = mp.mp_plan(h, 64, 64, 64)
    A, B, D = 0x10000, 0x20000000, 0x40000000  # never dereferenced
    g = lambda p, *a: lib.mp_gemm_with_plan(h.ptr, p, *a)
    assert g(ctypes.byref(plan), 64, 64, 64, A, 64, B, 64, None, 0, D, 64, 1.0, 0.0, None) == mp.MP_ERR_UNSUPPORTED
    assert g(None, 64, 64, 64, A, 64, B, 64, None, 0, D, 64, 1.0, 0.0, None) == mp.MP_ERR_INVALID_ARG
    assert g(ctypes.byref(plan), 64, 64, 64, A, 63, B, 64, None, 0, D, 64, 1.0, 0.0, None) == mp.MP_ERR_INVALID_ARG
    h.close()


def test_epilogue_word_and_bf16_output_checks():
    """mp_gemm_ex validates the epilogue word, bf16 D's alignment, and
    refuses C overlapping a bf16 D (different element types)."""
    lib = mp.library()
    h = _host()
    A, B, C, D = 0x10000, 0x20000000, 0x30000000, 0x40000000  # never dereferenced
    g = lambda epi, *a: lib.mp_gemm_ex(h.ptr, *a, epi, None)
    args = (64, 64, 64, A, 64, B, 64, C, 64, D, 64, 1.0, 0.5)
    assert g(0, *args) == mp.MP_ERR_UNSUPPORTED  # valid; planning-only handle
    assert g(mp.MP_ACT_GELU | mp.MP_EPI_OUT_BF16, *args) == mp.MP_ERR_UNSUPPORTED
    assert g(3, *args) == mp.MP_ERR_INVALID_ARG  # unknown activation
    assert g(0x200, *args) == mp.MP_ERR_INVALID_ARG  # unknown bit
    odd = (64, 64, 64, A, 64, B, 64, C, 64, D + 2, 64, 1.0, 0.5)
    assert g(mp.MP_EPI_OUT_BF16, *odd) == mp.MP_ERR_UNSUPPORTED  # 2-byte aligned bf16 D is fine
    assert g(0, *odd) == mp.MP_ERR_INVALID_ARG  # fp32 D needs 4-byte alignment
    assert g(mp.MP_EPI_OUT_BF16, *(64, 64, 64, A, 64, B, 64, C, 64, D + 1, 64, 1.0, 0.5)) == mp.MP_ERR_INVALID_ARG
    inplace = (64, 64, 64, A, 64, B, 64, D, 64, D, 64, 1.0, 0.5)
    assert g(0, *inplace) == mp.MP_ERR_UNSUPPORTED  # fp32 in place is allowed
    assert g(mp.MP_EPI_OUT_BF16, *inplace) == mp.MP_ERR_INVALID_ARG
    h.close()


def test_null_handle_and_host_init_errors():
    lib = mp.library()
    assert lib.mp_plan(None, 1, 1, 1, None) == mp.MP_ERR_INVALID_ARG
    assert lib.mp_destroy(None) == mp.MP_OK
    out = ctypes.c_void_p()
    assert lib.mp_init_host(ctypes.byref(out), None, None, 0) == mp.MP_ERR_INVALID_ARG
    assert lib.mp_init(None, 0, None) == mp.MP_ERR_INVALID_ARG


def test_mp_init_without_gpu_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    out = ctypes.c_void_p()
    st = mp.library().mp_init(ctypes.byref(out), 0, None)
    assert st in (mp.MP_ERR_UNSUPPORTED, mp.MP_ERR_CUDA) and not out.value


def test_b2b_argument_checks():
    """mp_gemm_b2b validates sizes, pointers, leading dimensions, overlaps and
    act0 before planning; valid calls on a planning-only handle report
    MP_ERR_UNSUPPORTED."""
    lib = mp.library()
    h = _host()
    A0, W0, C0, W1, C1, D1 = 0x10000, 0x20000000, 0x30000000, 0x40000000, 0x50000000, 0x60000000
    M, N0, N1, K0 = 100, 64, 96, 80

    def g(**kw):
        v = dict(M=M, N0=N0, N1=N1, K0=K0, A0=A0, lda0=K0, W0=W0, ldw0=N0, C0=C0, ldc0=N0, W1=W1, ldw1=N1,
                 C1=C1, ldc1=N1, D1=D1, ldd1=N1, a0=1.0, b0=0.5, a1=1.0, b1=0.5, act=0)
        v.update(kw)
        return lib.mp_gemm_b2b(h.ptr, v["M"], v["N0"], v["N1"], v["K0"], v["A0"], v["lda0"], v["W0"], v["ldw0"],
                               v["C0"], v["ldc0"], v["W1"], v["ldw1"], v["C1"], v["ldc1"], v["D1"], v["ldd1"],
                               v["a0"], v["b0"], v["a1"], v["b1"], v["act"], None)

    assert g() == mp.MP_ERR_UNSUPPORTED  # valid; no device
    assert g(act=2) == mp.MP_ERR_UNSUPPORTED
    assert g(M=0) == mp.MP_OK and g(N1=0) == mp.MP_OK  # no-ops
    for bad in (dict(M=-1), dict(K0=-1), dict(act=3), dict(act=-1), dict(D1=None), dict(ldd1=N1 - 1),
                dict(lda0=K0 - 1), dict(ldw0=N0 - 1), dict(ldw1=N1 - 1), dict(ldc0=N0 - 1), dict(ldc1=N1 - 1),
                dict(A0=None), dict(W1=None), dict(C0=None), dict(C1=None), dict(D1=D1 + 2), dict(A0=A0 + 1),
                dict(D1=C0), dict(D1=W1), dict(D1=A0), dict(C1=D1 + 4)):
        assert g(**bad) == mp.MP_ERR_INVALID_ARG, bad
    # C0 / C1 are not read when their beta is 0; W0, A0 not needed when K0 = 0.
    assert g(b0=0.0, C0=None, ldc0=0) == mp.MP_ERR_UNSUPPORTED
    assert g(b1=0.0, C1=None, ldc1=0) == mp.MP_ERR_UNSUPPORTED
    assert g(K0=0, A0=None, W0=None) == mp.MP_ERR_UNSUPPORTED
    # In place: C1 is D1 (same pointer and ld).
    assert g(C1=D1) == mp.MP_ERR_UNSUPPORTED
    # N0 past one accumulator: valid (two launches); still no device here.
    assert g(N0=257, ldw0=257, ldc0=257) == mp.MP_ERR_UNSUPPORTED
    h.close()


def test_b2b_form_choice():
    """The fused kernel unless two launches are clearly faster; N0 > 256 as
    two launches; a forced mode wins (and a forced fused form refuses
    N0 > 256).  With the measured table (the default) the choice follows
    what GB300 measured on cold operands: 256 -> 64 -> 256 pairs ran faster
    fused at every M (M = 1000: 7.5 against 8.9 us; M = 75264: 27.3 against
    30.8 us), 768 -> 256 -> 768 pairs faster as two launches (M = 2136: 13.0
    against 14.4 us)."""
    cal = _host()
    mp.mp_load_calibration(cal, os.path.join(ROOT, "micro_polymerization_gb300", "calib", "gb300.txt"))
    for M in (1000, 100352):
        assert mp.mp_plan_b2b(cal, M, 64, 256, 256).mode == mp.MP_B2B_FUSED
    for M in (256, 2048):
        assert mp.mp_plan_b2b(cal, M, 256, 768, 768).mode == mp.MP_B2B_TWO_LAUNCH
    # Every problem of the two fused-pair workloads takes the form its
    # workload ran faster in as a whole (0.750 ms all fused against 0.846 ms
    # as two launches; 0.813 ms as two launches against 0.936 ms fused).
    from micro_polymerization_gb300 import workloads as wl
    for name, mode in (("b2b_1x1", mp.MP_B2B_FUSED), ("b2b_adapter", mp.MP_B2B_TWO_LAUNCH)):
        for b in wl.B2B_WORKLOADS[name]():
            assert mp.mp_plan_b2b(cal, b.M, b.N0, b.N1, b.K0).mode == mode, (name, b.M)
    cal.close()
    h = _host()  # the analytic model
    assert mp.mp_plan_b2b(h, 100352, 64, 256, 256).mode == mp.MP_B2B_FUSED
    assert mp.mp_plan_b2b(h, 2048, 256, 768, 768).mode == mp.MP_B2B_FUSED
    assert mp.mp_plan_b2b(h, 2048, 384, 768, 768).mode == mp.MP_B2B_TWO_LAUNCH
    for M in (1, 512, 4096, 100352):
        p = mp.mp_plan_b2b(h, M, 64, 256, 256)
        assert p.two_launch_cost_us > 0 and p.cost_us > 0
    mp.mp_set_b2b_mode(h, mp.MP_B2B_FUSED)
    assert mp.mp_plan_b2b(h, 256, 256, 768, 768).mode == mp.MP_B2B_FUSED
    with pytest.raises(mp.MPError):
        mp.mp_plan_b2b(h, 2048, 384, 768, 768)
    mp.mp_set_b2b_mode(h, mp.MP_B2B_TWO_LAUNCH)
    assert mp.mp_plan_b2b(h, 100352, 64, 256, 256).mode == mp.MP_B2B_TWO_LAUNCH
    with pytest.raises(mp.MPError):
        mp.mp_set_b2b_mode(h, 3)
    h.close()


def test_b2b_plan_rules():
    h = _host()
    for M, N0, N1, K0 in [(1, 1, 1, 1), (1000, 256, 768, 768), (128 * 400, 64, 256, 256), (256, 128, 4096, 64),
                          (300, 96, 520, 0), (77, 0, 300, 50), (5000, 200, 100, 3000)]:
        p = mp.mp_plan_b2b(h, M, N0, N1, K0)
        assert p.n0p == -(-N0 // 64) * 64 and p.n0p <= 256
        assert p.bn1 % 64 == 0 and 64 <= p.bn1 <= 256 and p.chunks * p.bn1 >= N1 > (p.chunks - 1) * p.bn1
        assert p.mblocks == -(-M // 128)
        groups = -(-p.chunks // p.cpg)
        assert 1 <= p.cpg <= p.chunks and p.units == p.mblocks * groups
        assert p.grid == min(p.units, 148)
        assert 2 <= p.num_stages <= 8 and p.smem_bytes <= 232448
        ring_need = max((16384 + p.n0p * 128) if (K0 > 0 and N0 > 0) else 0, p.bn1 * 128)
        assert p.stage_bytes == ring_need and p.stage_bytes % 8192 == 0
        assert p.cost_us > 0
    # A costly first GEMM with many row blocks: no recomputation of D0.
    p = mp.mp_plan_b2b(h, 128 * 1000, 256, 1024, 4096)
    assert p.cpg == p.chunks and p.units == 1000
    # One row block, many chunks, a cheap first GEMM: chunks spread over SMs.
    p = mp.mp_plan_b2b(h, 128, 128, 8192, 64)
    assert p.cpg < p.chunks and p.units > 1
    p = mp.mp_plan_b2b(h, 10, 257, 10, 10)  # wider than one accumulator: two launches
    assert p.mode == mp.MP_B2B_TWO_LAUNCH and p.units == 0
    with pytest.raises(mp.MPError):
        mp.mp_plan_b2b(h, -1, 64, 10, 10)
    h.close()


def test_conv_argument_checks():
    lib = mp.library()
    h = _host()
    X, F, Cin, D = 0x10000, 0x20000000, 0x30000000, 0x40000000
    base = dict(N=2, H=8, W=9, C=16, K=24, R=3, S=3, ph=1, pw=1, X=X, F=F, Cin=Cin, ldc=24, D=D, ldd=24,
                a=1.0, b=0.5)

    def g(**kw):
        v = dict(base)
        v.update(kw)
        return lib.mp_conv2d(h.ptr, v["N"], v["H"], v["W"], v["C"], v["K"], v["R"], v["S"], v["ph"], v["pw"],
                             v["X"], v["F"], v["Cin"], v["ldc"], v["D"], v["ldd"], v["a"], v["b"], None)

    assert g() == mp.MP_ERR_UNSUPPORTED  # valid; no device
    for empty in (dict(N=0), dict(K=0), dict(H=1, ph=0), dict(W=2, pw=0)):
        assert g(**empty) == mp.MP_OK, empty
    for bad in (dict(N=-1), dict(C=-1), dict(R=0), dict(S=0), dict(ph=-1), dict(D=None), dict(ldd=23),
                dict(X=None), dict(F=None), dict(Cin=None), dict(ldc=23), dict(D=D + 2), dict(X=X + 1),
                dict(D=X), dict(D=F), dict(Cin=D + 4)):
        assert g(**bad) == mp.MP_ERR_INVALID_ARG, bad
    assert g(b=0.0, Cin=None, ldc=0) == mp.MP_ERR_UNSUPPORTED  # Cin not read
    assert g(C=0, X=None, F=None) == mp.MP_ERR_UNSUPPORTED    # no operand read
    assert g(Cin=D) == mp.MP_ERR_UNSUPPORTED                  # in place
    h.close()


def test_conv_plan_rules():
    h = _host()
    for (N, H, W, C, K, R, S, ph, pw) in [(1, 1, 1, 1, 1, 1, 1, 0, 0), (32, 80, 80, 64, 64, 3, 3, 1, 1),
                                           (5, 5, 5, 512, 512, 3, 3, 1, 1), (2, 7, 9, 16, 24, 3, 3, 1, 1),
                                           (3, 30, 17, 12, 20, 5, 5, 2, 2), (1, 224, 224, 3, 64, 1, 1, 0, 0)]:
        p = mp.mp_plan_conv(h, N, H, W, C, K, R, S, ph, pw)
        P, Q = H + 2 * ph - R + 1, W + 2 * pw - S + 1
        assert 1 <= p.wb * p.hb * p.nb <= 128 and p.nb <= max(N, 128 // (p.wb * p.hb))
        assert p.tiles_q == -(-Q // p.wb) and p.tiles_p == -(-P // p.hb) and p.tiles_n == -(-N // p.nb)
        assert p.bn in (64, 128, 256) and p.tiles_k == -(-K // p.bn)
        assert p.tiles == p.tiles_q * p.tiles_p * p.tiles_n * p.tiles_k
        assert 1 <= p.splits <= max(1, p.ksteps) and p.units == p.tiles * p.splits and p.grid == min(p.units, 148)
        assert p.splits == 1 or p.tiles * p.splits * 128 * p.bn <= 16 << 20  # the workspace
        assert p.ksteps == R * S * -(-C // 64)
        assert 0 < p.useful <= 1 and p.useful == pytest.approx(N * P * Q / (p.tiles_q * p.wb * p.tiles_p * p.hb
                                                                             * p.tiles_n * p.nb))
        assert 2 <= p.num_stages <= 8 and p.smem_bytes <= 232448 and p.stage_bytes == 16384 + 128 * p.bn
    # Small images: tiles take several images rather than padding one image,
    # with sides that fit the image when that wastes fewer rows.
    p = mp.mp_plan_conv(h, 32, 7, 7, 512, 512)
    assert p.nb > 1 and p.useful > 0.85
    p = mp.mp_plan_conv(h, 20, 5, 5, 512, 512)
    assert p.useful > 0.9
    # Few tiles and a long K loop: split K.
    assert mp.mp_plan_conv(h, 1, 7, 7, 512, 512).splits > 1
    p = mp.mp_plan_conv(h, 2, 0, 5, 8, 8)  # empty output
    assert p.units == 0 and p.grid == 0
    with pytest.raises(mp.MPError):
        mp.mp_plan_conv(h, 1, 5, 5, 8, 8, 0, 3)
    h.close()


def test_grouped_argument_checks_and_plan():
    lib = mp.library()
    h = _host()
    P = mp.MpGemmProblem

    def call(probs):
        arr = (P * max(1, len(probs)))(*probs)
        return lib.mp_gemm_grouped(h.ptr, len(probs), arr, None)

    a0 = P(100, 96, 80, 0x10000, 80, 0x100000, 96, None, 0, 0x200000, 96, 1.0, 0.0)
    a1 = P(33, 17, 5, 0x300000, 5, 0x310000, 17, 0x320000, 17, 0x330000, 17, 1.0, 0.5)
    assert call([a0, a1]) == mp.MP_ERR_UNSUPPORTED  # valid; no device
    assert call([]) == mp.MP_OK
    assert call([P(0, 5, 5, 0, 5, 0, 5, None, 0, 0, 5, 1.0, 0.0)]) == mp.MP_OK  # only empty problems
    # One problem breaking mp_gemm's rules.
    assert call([a0, P(10, 10, 10, 0x10000, 9, 0x20000, 10, None, 0, 0x500000, 10, 1.0, 0.0)]) == mp.MP_ERR_INVALID_ARG
    # Output of one problem overlapping another's output or operands.
    clash_d = P(10, 10, 10, 0x600000, 10, 0x610000, 10, None, 0, 0x200000 + 4 * 96, 10, 1.0, 0.0)
    assert call([a0, clash_d]) == mp.MP_ERR_INVALID_ARG
    clash_a = P(10, 10, 10, 0x600000, 10, 0x610000, 10, None, 0, 0x10000 + 64, 10, 1.0, 0.0)
    assert call([a0, clash_a]) == mp.MP_ERR_INVALID_ARG
    assert lib.mp_gemm_grouped(h.ptr, -1, None, None) == mp.MP_ERR_INVALID_ARG
    assert lib.mp_gemm_grouped(h.ptr, 2, None, None) == mp.MP_ERR_INVALID_ARG
    # Plan: one tile width, the group's tiles, one launch per 48 problems.
    shapes = [(int(m), 2048, 1024) for m in np.random.default_rng(0).integers(1, 513, 100)]
    p = mp.mp_plan_grouped(h, shapes)
    assert p.bn in (64, 128, 256) and p.launches == 3
    assert p.units == sum(-(-m // 128) * -(-n // p.bn) for m, n, _ in shapes)
    assert p.smem_bytes <= 232448 and p.stage_bytes == 16384 + 128 * p.bn and p.cost_us > 0
    h.close()

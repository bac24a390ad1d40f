"""GPU parity of the fused back-to-back GEMM (mp_gemm_b2b) against the fp64
oracle (BOLT summary, persistent kernel (GEMM/Conv) fusion).

Bound, element by element (oracle.b2b_bound): the first GEMM's stated bound
carried through the activation and the second GEMM, one bf16 rounding of the
on-chip D0, and the second GEMM's own stated bound."""
import numpy as np
import pytest
import torch

import micro_polymerization_gb300 as mp
import oracle
from micro_polymerization_gb300 import workloads as wl

from gpu_util import handle

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.fixture(autouse=True)
def fused_form():
    """These tests check the fused kernel itself: force it (the automatic
    choice would take the two-launch form for small M), then restore."""
    mp.mp_set_b2b_mode(handle(), mp.MP_B2B_FUSED)
    yield
    mp.mp_set_b2b_mode(handle(), mp.MP_B2B_AUTO)


def _bits(t):
    return wl.bf16_bits(t.cpu())


def run_b2b(b, D1=None, c1_is_d1=False, rows=None):
    """Run one problem; returns (D1 on the CPU, oracle D1, bound) over `rows`."""
    A0, W0, C0, W1, C1 = wl.make_b2b_operands(b)
    d = [t.to(DEV) if t is not None else None for t in (A0, W0, C0, W1, C1)]
    if D1 is None:
        D1 = torch.full((b.M, b.N1), float("nan"), device=DEV)
    if c1_is_d1:
        D1.copy_(d[4])
        d[4] = D1
    mp.mp_gemm_b2b(handle(), d[0], d[1], d[2], d[3], d[4], D1, b.alpha0, b.beta0, b.alpha1, b.beta1, b.act0)
    torch.cuda.synchronize()
    assert mp.mp_check(handle()) == 0
    out = D1.cpu()
    sel = slice(None) if rows is None else rows
    A0b = _bits(A0)[sel]
    C0n = C0.numpy()[sel] if C0 is not None else None
    C1n = C1.numpy()[sel] if C1 is not None else None
    args = (A0b, _bits(W0), C0n, _bits(W1), C1n, b.alpha0, b.beta0, b.alpha1, b.beta1)
    ref, d0 = oracle.b2b(*args, b.act0)
    bound = oracle.b2b_bound(*args, b.act0, d0)
    return out.numpy()[sel], ref, bound


def check(b, **kw):
    got, ref, bound = run_b2b(b, **kw)
    ok, worst = oracle.within_b2b(got, ref, bound)
    assert ok, f"{b}: worst err/bound {worst:.3g}"
    return worst


@pytest.mark.parametrize("act", [0, 1, 2])
@pytest.mark.parametrize("M,N0,N1,K0", [(300, 96, 520, 200), (129, 256, 768, 768), (1, 64, 64, 64),
                                        (200, 17, 33, 5), (257, 192, 300, 130)])
def test_b2b_parity_ragged(M, N0, N1, K0, act):
    check(wl.B2B(M, N0, N1, K0, alpha0=1.25, beta0=0.5, alpha1=0.75, beta1=-0.5, act0=act, seed=M + N0 + N1 + K0))


def test_b2b_beta_zero_and_no_c():
    check(wl.B2B(333, 128, 256, 384, act0=1, seed=9))


def test_b2b_many_units_per_cta():
    """More row blocks than SMs: each CTA runs several units in turn, reusing
    its D0 block, ring and accumulators (sampled rows, all row blocks hit)."""
    b = wl.B2B(128 * 400 + 37, 64, 256, 128, alpha0=1.0, beta0=0.25, alpha1=1.0, beta1=0.5, act0=2, seed=4)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(0, b.M, 97), rng.integers(0, b.M, 2000), np.arange(b.M - 40, b.M)]))
    got, ref, bound = run_b2b(b, rows=rows)
    ok, worst = oracle.within_b2b(got, ref, bound)
    assert ok, worst


def test_b2b_recompute_groups():
    """Few row blocks and many chunks of D1: the planner splits the chunks of
    a row block over several units, each recomputing D0."""
    b = wl.B2B(256, 128, 4096, 64, alpha0=1.0, beta0=0.0, alpha1=1.0, beta1=0.0, act0=0, seed=5)
    plan = mp.mp_plan_b2b(handle(), b.M, b.N0, b.N1, b.K0)
    assert plan.cpg < plan.chunks
    check(b)


def test_b2b_degenerate_k0_and_n0():
    # K0 = 0: D0 = act(beta0 * C0).
    check(wl.B2B(150, 64, 200, 0, alpha0=2.0, beta0=1.5, alpha1=1.0, beta1=0.5, act0=1, seed=6))
    # N0 = 0: D1 = beta1 * C1.
    b = wl.B2B(150, 0, 200, 64, beta1=0.5, seed=7)
    A0, W0, C0, W1, C1 = wl.make_b2b_operands(b)
    D1 = torch.full((b.M, b.N1), float("nan"), device=DEV)
    mp.mp_gemm_b2b(handle(), A0.to(DEV), W0.to(DEV), None, W1.to(DEV), C1.to(DEV), D1, 1.0, 0.0, 1.0, 0.5)
    torch.cuda.synchronize()
    assert torch.equal(D1.cpu(), 0.5 * C1)


def test_b2b_unaligned_d1_and_in_place_c1():
    b = wl.B2B(190, 80, 301, 100, alpha0=1.0, beta0=0.0, alpha1=1.0, beta1=1.0, act0=0, seed=8)
    base = torch.full((b.M * (b.N1 + 1) + 1,), float("nan"), device=DEV)
    D1 = base[1:1 + b.M * (b.N1 + 1)].view(b.M, b.N1 + 1)[:, :b.N1]  # odd pitch, 4-byte offset
    check(b, D1=D1)
    check(b, c1_is_d1=True)


def test_b2b_identity_w1_matches_fused_epilogue_gemm():
    """W1 = I and beta1 = 0: D1 is D0 rounded to bf16, i.e. exactly what
    mp_gemm_ex with the same activation and a bf16 D writes."""
    M, K0, N0 = 300, 200, 128
    b = wl.B2B(M, N0, N0, K0, alpha0=1.0, beta0=0.5, act0=2, seed=10)
    A0, W0, C0, _, _ = wl.make_b2b_operands(b)
    eye = torch.eye(N0, dtype=torch.bfloat16, device=DEV)
    D1 = torch.empty(M, N0, device=DEV)
    mp.mp_gemm_b2b(handle(), A0.to(DEV), W0.to(DEV), C0.to(DEV), eye, None, D1, 1.0, 0.5, 1.0, 0.0, 2)
    # The plain GEMM on a 128 x 128 normal tile without split-K: the same
    # K-step sequence and epilogue arithmetic as the fused kernel's first GEMM.
    _, ks = mp.mp_get_hw(handle())
    k128 = [i for i, k in enumerate(ks) if k.um == 128 and k.un == 128 and not k.swap and not k.pair][0]
    Dx = torch.empty(M, N0, device=DEV, dtype=torch.bfloat16)
    mp.mp_force_plan(handle(), k128, 1)
    try:
        mp.mp_gemm_ex(handle(), A0.to(DEV), W0.to(DEV), C0.to(DEV), Dx, 1.0, 0.5, act=2)
        torch.cuda.synchronize()
    finally:
        mp.mp_force_plan(handle(), -1, 0)
    got, want = D1.cpu().double(), Dx.float().cpu().double()
    # Products with I are exact, so D1 is the bf16 D0 itself; allow one bf16
    # rounding step in case the two launches accumulate K in another order.
    assert torch.all((got - want).abs() <= want.abs() * 2.0 ** -7)
    assert (got == want).double().mean() > 0.99


def test_b2b_adapter_workload_sampled():
    """Full-size problems of the b2b_adapter workload (the largest M, and a
    mid-size one) on sampled rows, with the bench's parameters."""
    bs = sorted(wl.b2b_adapter(), key=lambda b: b.M)
    rng = np.random.default_rng(1)
    for b in (bs[-1], bs[len(bs) // 2]):
        rows = np.unique(np.concatenate([[0, b.M - 1], rng.integers(0, b.M, 48)]))
        got, ref, bound = run_b2b(b, rows=rows)
        ok, worst = oracle.within_b2b(got, ref, bound)
        assert ok, (b, worst)


@pytest.mark.parametrize("shape", [(300, 96, 520, 200, 2), (129, 256, 768, 768, 1), (200, 17, 33, 5, 0),
                                   (150, 64, 200, 0, 1), (4096, 256, 768, 768, 1)])
def test_b2b_two_launch_form(shape):
    """The two-launch form (bf16 D0 in the handle's scratch buffer) meets the
    same bound."""
    M, N0, N1, K0, act = shape
    mp.mp_set_b2b_mode(handle(), mp.MP_B2B_TWO_LAUNCH)
    check(wl.B2B(M, N0, N1, K0, alpha0=1.25, beta0=0.5, alpha1=0.75, beta1=-0.5, act0=act, seed=M + K0))


def test_b2b_auto_choice_runs_the_planned_form():
    """AUTO takes the form mp_plan_b2b reports: the fused kernel for a
    256 -> 64 -> 256 pair, two launches for a 768 -> 256 -> 768 pair of
    small M (measured faster that way) and for a D0 wider than one
    accumulator; each within the bound."""
    mp.mp_set_b2b_mode(handle(), mp.MP_B2B_AUTO)
    wide = wl.B2B(300, 384, 200, 160, alpha0=1.0, beta0=0.5, alpha1=1.0, beta1=0.5, act0=2, seed=21)
    large = wl.B2B(128 * 400, 64, 256, 256, act0=1, seed=22)
    adapter = wl.B2B(2048, 256, 768, 768, act0=1, seed=23)
    assert mp.mp_plan_b2b(handle(), wide.M, wide.N0, wide.N1, wide.K0).mode == mp.MP_B2B_TWO_LAUNCH
    assert mp.mp_plan_b2b(handle(), large.M, large.N0, large.N1, large.K0).mode == mp.MP_B2B_FUSED
    assert mp.mp_plan_b2b(handle(), adapter.M, adapter.N0, adapter.N1, adapter.K0).mode == mp.MP_B2B_TWO_LAUNCH
    check(wide)
    check(adapter)
    rows = np.arange(0, large.M, 331)
    got, ref, bound = run_b2b(large, rows=rows)
    ok, worst = oracle.within_b2b(got, ref, bound)
    assert ok, worst


def test_b2b_two_launch_form_allocates_nothing():
    """The two-launch form keeps D0 at the end of the handle's staging area:
    a call with unaligned A0, W0 and W1 (staged in front of D0) meets the
    bound, and repeating it leaves the device's free memory unchanged."""
    mp.mp_set_b2b_mode(handle(), mp.MP_B2B_TWO_LAUNCH)
    b = wl.B2B(300, 100, 77, 130, alpha0=1.0, beta0=0.5, alpha1=1.0, beta1=0.5, act0=1, seed=31)
    A0, W0, C0, W1, C1 = wl.make_b2b_operands(b)
    d = [t.to(DEV) for t in (A0, W0, C0, W1, C1)]
    D1 = torch.empty(b.M, b.N1, device=DEV)
    for call in range(2):
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info(0)[0]
        mp.mp_gemm_b2b(handle(), d[0], d[1], d[2], d[3], d[4], D1, b.alpha0, b.beta0, b.alpha1, b.beta1,
                       b.act0)
        torch.cuda.synchronize()
        assert mp.mp_check(handle()) == 0
        assert torch.cuda.mem_get_info(0)[0] == free0, f"call {call + 1} changed free device memory"
    args = (_bits(A0), _bits(W0), C0.numpy(), _bits(W1), C1.numpy(), b.alpha0, b.beta0, b.alpha1, b.beta1)
    ref, d0 = oracle.b2b(*args, b.act0)
    ok, worst = oracle.within_b2b(D1.cpu().numpy(), ref, oracle.b2b_bound(*args, b.act0, d0))
    assert ok, worst

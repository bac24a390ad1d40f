"""GPU parity of the implicit-GEMM convolution (mp_conv2d) against the fp64
oracle.  Bound, element by element, as for a GEMM (the convolution is the GEMM
over its im2col matrix): |D - D_ref| <= 2e-3 * (sum |X||F| + |beta Cin|)."""
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


def run_conv(c, X=None, F=None, Cin=None, D=None, in_place=False):
    if X is None:
        X, F, Cin = wl.make_conv_operands(c)
    Xd, Fd = X.to(DEV), F.to(DEV)
    Cd = Cin.to(DEV) if Cin is not None else None
    if D is None:
        D = torch.full((c.N, c.P, c.Q, c.K), float("nan"), device=DEV)
    if in_place:
        D.copy_(Cd)
        Cd = D
    mp.mp_conv2d(handle(), Xd, Fd, Cd, D, c.alpha, c.beta, c.pad_h, c.pad_w)
    torch.cuda.synchronize()
    assert mp.mp_check(handle()) == 0
    return D.cpu(), X, F, Cin


def check(c, **kw):
    D, X, F, Cin = run_conv(c, **kw)
    Cn = Cin.numpy() if Cin is not None else None
    ref = oracle.conv2d_nhwc(_bits(X), _bits(F), Cn, c.alpha, c.beta, c.pad_h, c.pad_w)
    mag = oracle.conv2d_magnitude(_bits(X), _bits(F), Cn, c.beta, c.pad_h, c.pad_w)
    ok, worst = oracle.within_bound(D.numpy().reshape(-1, c.K), ref.reshape(-1, c.K), mag.reshape(-1, c.K))
    assert ok, f"{c}: worst {worst:.3g}"


@pytest.mark.parametrize("shape", [
    (2, 7, 9, 16, 24, 3, 3, 1, 1),      # C < 64, K < 64, ragged tiles
    (3, 20, 20, 64, 64, 3, 3, 1, 1),
    (1, 40, 45, 128, 128, 3, 3, 1, 1),
    (5, 5, 5, 512, 512, 3, 3, 1, 1),    # small images: boxes over several images
    (2, 10, 10, 256, 256, 3, 3, 1, 1),
    (2, 8, 8, 12, 20, 3, 3, 1, 1),      # C, K not multiples of 8: staged operands
    (2, 9, 11, 40, 30, 3, 3, 1, 1),     # K % 4 != 0: plain stores
    (2, 6, 7, 80, 96, 5, 5, 2, 2),
    (1, 12, 13, 72, 64, 1, 3, 0, 2),    # asymmetric filter and padding
    (4, 14, 14, 100, 130, 1, 1, 0, 0),  # 1x1
])
def test_conv_parity(shape):
    N, H, W, C, K, R, S, ph, pw = shape
    check(wl.Conv(N, H, W, C, K, R, S, ph, pw, alpha=1.25, beta=0.5, seed=sum(shape)))


@pytest.mark.parametrize("shape", [(20, 5, 5, 512, 512), (9, 9, 9, 256, 256), (7, 7, 7, 128, 96), (3, 6, 10, 64, 64)])
def test_conv_exact_fit_boxes(shape):
    """Small images: boxes whose sides divide the image (not powers of two,
    fewer than 128 rows, pixel-by-pixel stores) within the bound."""
    N, H, W, C, K = shape
    c = wl.Conv(N, H, W, C, K, alpha=1.25, beta=0.5, seed=H * W + C)
    check(c)


def test_conv_some_plan_uses_an_exact_fit_box():
    boxes = [mp.mp_plan_conv(handle(), *s) for s in [(20, 5, 5, 512, 512), (9, 9, 9, 256, 256), (7, 7, 7, 128, 96)]]
    assert any(p.wb * p.hb * p.nb < 128 for p in boxes), [(p.wb, p.hb, p.nb) for p in boxes]


def test_conv_integer_exact():
    """Integer data: every partial sum is exact in fp32, so bitwise equal."""
    for (N, H, W, C, K) in [(2, 9, 7, 24, 40), (3, 5, 5, 128, 64), (1, 33, 17, 64, 192)]:
        c = wl.Conv(N, H, W, C, K, alpha=1.0, beta=1.0, seed=N * H + K)
        gen = torch.Generator().manual_seed(c.seed)
        X = torch.randint(-3, 4, (N, H, W, C), generator=gen).to(torch.bfloat16)
        F = torch.randint(-3, 4, (3, 3, C, K), generator=gen).to(torch.bfloat16)
        Cin = torch.randint(-3, 4, (N, H, W, K), generator=gen).to(torch.float32)
        D, _, _, _ = run_conv(c, X, F, Cin)
        ref = oracle.conv2d_nhwc(_bits(X), _bits(F), Cin.numpy(), 1.0, 1.0)
        assert np.array_equal(D.numpy().astype(np.float64), ref), (N, H, W, C, K)


def test_conv_split_k_parity_and_determinism():
    """Few tiles and a long K loop: the plan splits K; partials are summed in
    split order, so two runs give the same bits."""
    for shape in [(1, 7, 7, 512, 512), (2, 5, 6, 256, 320), (1, 9, 9, 300, 72)]:
        N, H, W, C, K = shape
        c = wl.Conv(N, H, W, C, K, alpha=1.5, beta=0.5, seed=N + C)
        plan = mp.mp_plan_conv(handle(), N, H, W, C, K)
        assert plan.splits > 1, (shape, plan.splits)
        check(c)
        D1, _, _, _ = run_conv(c)
        D2, _, _, _ = run_conv(c)
        assert torch.equal(D1, D2)


def test_conv_c_zero_and_in_place():
    c = wl.Conv(2, 6, 6, 0, 64, alpha=1.0, beta=0.5, seed=3)
    X = torch.zeros(2, 6, 6, 0, dtype=torch.bfloat16)
    F = torch.zeros(3, 3, 0, 64, dtype=torch.bfloat16)
    Cin = torch.rand(2, 6, 6, 64)
    D, _, _, _ = run_conv(c, X, F, Cin)
    assert torch.equal(D, 0.5 * Cin)
    check(wl.Conv(2, 11, 13, 64, 128, alpha=1.0, beta=1.0, seed=4), in_place=True)


def test_conv_matches_gemm_on_im2col():
    """The same layer through mp_gemm on the explicit im2col matrix (the
    GEMM-based convolution of the pages): both within the bound of one
    oracle, and close to each other."""
    c = wl.Conv(4, 12, 12, 64, 64, alpha=1.0, beta=0.0, seed=9)
    D, X, F, _ = run_conv(c)
    A = torch.from_numpy(oracle.im2col_nhwc(_bits(X), 3, 3).view(np.int16)).view(torch.bfloat16)
    B = F.reshape(9 * c.C, c.K)
    Dg = torch.empty(A.shape[0], c.K, device=DEV)
    mp.mp_gemm(handle(), A.to(DEV), B.to(DEV), None, Dg, 1.0, 0.0)
    torch.cuda.synchronize()
    ref = oracle.gemm(_bits(A), _bits(B))
    mag = oracle.magnitude(_bits(A), _bits(B))
    for got in (D.reshape(-1, c.K), Dg.cpu()):
        ok, worst = oracle.within_bound(got.numpy(), ref, mag)
        assert ok, worst


def test_conv_workload_sample():
    """A few layers of the dynamic-resolution workload, sampled outputs."""
    rng = np.random.default_rng(0)
    for c in wl.conv_resolution()[:6]:
        D, X, F, Cin = run_conv(c)
        # Full-oracle check on two images (the rest by the same code path).
        n = min(c.N, 2)
        ref = oracle.conv2d_nhwc(_bits(X[:n]), _bits(F), None, c.alpha, 0.0)
        mag = oracle.conv2d_magnitude(_bits(X[:n]), _bits(F))
        ok, worst = oracle.within_bound(D[:n].numpy().reshape(-1, c.K), ref.reshape(-1, c.K),
                                        mag.reshape(-1, c.K))
        assert ok, (c, worst)
        assert torch.isfinite(D).all()

"""Seeded synthetic workloads: GEMM shape lists and operand generators.

This module holds no GEMM arithmetic.  It only draws shapes and random
operands, so that the GPU library and the CPU oracle can be fed the very same
bytes.  The pages measure on DeepBench GEMMs and on shape ranges taken from
real Transformer and CNN models (MikPoly summary, section 5 "Evaluation");
none of those sets is available here, so each workload below is a seeded
stand-in with the shapes and value ranges the workload describes.

Operand recipe (every workload): A[M,K] and B[K,N] are drawn as fp32 uniform
on [-1, 1) from ``torch.Generator().manual_seed(seed)`` and rounded to bf16
(round to nearest even); C[M,N] is fp32 uniform on [-1, 1) from the next
seed; D is fp32.  Shape lists are drawn with ``numpy.random.default_rng``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Gemm:
    """One GEMM problem: D[M,N] = alpha*A[M,K]*B[K,N] + beta*C[M,N] (batch copies)."""
    M: int
    N: int
    K: int
    alpha: float = 1.0
    beta: float = 0.0
    batch: int = 1
    seed: int = 0

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K * self.batch

    def min_bytes(self, d_bytes: int = 4) -> int:
        """Each operand read once, D written once: the algorithmic traffic
        (d_bytes per element of D: 4 for fp32, 2 for bf16)."""
        per = 2 * self.M * self.K + 2 * self.K * self.N + d_bytes * self.M * self.N
        if self.beta != 0.0:
            per += 4 * self.M * self.N
        return per * self.batch


def _uniform(shape, gen: torch.Generator, device) -> torch.Tensor:
    return torch.rand(shape, generator=gen, device=device, dtype=torch.float32).mul_(2.0).sub_(1.0)


def make_operands(g: Gemm, device="cpu"):
    """Operands of one problem, seeded by ``g.seed``.

    Returns (A bf16 [batch,M,K] or [M,K], B bf16 [batch,K,N] or [K,N],
    C fp32 like D or None when beta == 0).
    """
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(g.seed))
    lead = (g.batch,) if g.batch > 1 else ()
    A = _uniform(lead + (g.M, g.K), gen, dev).to(torch.bfloat16)
    B = _uniform(lead + (g.K, g.N), gen, dev).to(torch.bfloat16)
    C = None
    if g.beta != 0.0:
        gen.manual_seed(int(g.seed) + 1)
        C = _uniform(lead + (g.M, g.N), gen, dev)
    return A, B, C


def integer_operands(M: int, N: int, K: int, seed: int, lo: int = -4, hi: int = 4, device="cpu"):
    """Integer-valued bf16 A, B and fp32 C in [lo, hi] (exact in bf16 and in sums)."""
    gen = torch.Generator(device=torch.device(device))
    gen.manual_seed(int(seed))
    A = torch.randint(lo, hi + 1, (M, K), generator=gen, device=device).to(torch.bfloat16)
    B = torch.randint(lo, hi + 1, (K, N), generator=gen, device=device).to(torch.bfloat16)
    C = torch.randint(lo, hi + 1, (M, N), generator=gen, device=device).to(torch.float32)
    return A, B, C


@dataclasses.dataclass(frozen=True)
class B2B:
    """Back-to-back GEMMs: D1[M,N1] = alpha1 * act0(alpha0 * A0[M,K0] W0[K0,N0]
    + beta0 * C0[M,N0]) W1[N0,N1] + beta1 * C1[M,N1]."""
    M: int
    N0: int
    N1: int
    K0: int
    alpha0: float = 1.0
    beta0: float = 0.0
    alpha1: float = 1.0
    beta1: float = 0.0
    act0: int = 0
    seed: int = 0

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N0 * self.K0 + 2 * self.M * self.N1 * self.N0

    def min_bytes(self) -> int:
        """A0, W0, W1 (and C0, C1 when read) once, D1 written once; D0 never
        leaves the chip."""
        b = 2 * self.M * self.K0 + 2 * self.K0 * self.N0 + 2 * self.N0 * self.N1 + 4 * self.M * self.N1
        if self.beta0 != 0.0:
            b += 4 * self.M * self.N0
        if self.beta1 != 0.0:
            b += 4 * self.M * self.N1
        return b


def make_b2b_operands(b: B2B, device="cpu"):
    """(A0, W0, W1) bf16 and (C0, C1) fp32 or None, uniform [-1, 1), seeded by b.seed."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(b.seed))
    A0 = _uniform((b.M, b.K0), gen, dev).to(torch.bfloat16)
    W0 = _uniform((b.K0, b.N0), gen, dev).to(torch.bfloat16)
    W1 = _uniform((b.N0, b.N1), gen, dev).to(torch.bfloat16)
    gen.manual_seed(int(b.seed) + 1)
    C0 = _uniform((b.M, b.N0), gen, dev) if b.beta0 != 0.0 else None
    C1 = _uniform((b.M, b.N1), gen, dev) if b.beta1 != 0.0 else None
    return A0, W0, C0, W1, C1


@dataclasses.dataclass(frozen=True)
class Conv:
    """Stride-1 2-D convolution, NHWC: D[N,P,Q,K] = alpha * conv(X[N,H,W,C],
    F[R,S,C,K]) + beta * Cin, P = H + 2 pad_h - R + 1, Q likewise."""
    N: int
    H: int
    W: int
    C: int
    K: int
    R: int = 3
    S: int = 3
    pad_h: int = 1
    pad_w: int = 1
    alpha: float = 1.0
    beta: float = 0.0
    seed: int = 0

    @property
    def P(self) -> int:
        return self.H + 2 * self.pad_h - self.R + 1

    @property
    def Q(self) -> int:
        return self.W + 2 * self.pad_w - self.S + 1

    @property
    def flops(self) -> int:
        return 2 * self.N * self.P * self.Q * self.K * self.R * self.S * self.C

    def as_gemm(self) -> "Gemm":
        """The GEMM a GEMM-based convolution runs: [N*P*Q, R*S*C] x [R*S*C, K]."""
        return Gemm(self.N * self.P * self.Q, self.K, self.R * self.S * self.C, self.alpha, self.beta, seed=self.seed)

    def min_bytes(self) -> int:
        """X and F read once, D written once (and Cin read when beta != 0)."""
        b = 2 * self.N * self.H * self.W * self.C + 2 * self.R * self.S * self.C * self.K
        b += 4 * self.N * self.P * self.Q * self.K * (2 if self.beta != 0.0 else 1)
        return b


def make_conv_operands(c: Conv, device="cpu"):
    """(X bf16 [N,H,W,C], F bf16 [R,S,C,K], Cin fp32 [N,P,Q,K] or None), uniform [-1, 1)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(c.seed))
    X = _uniform((c.N, c.H, c.W, c.C), gen, dev).to(torch.bfloat16)
    F = _uniform((c.R, c.S, c.C, c.K), gen, dev).to(torch.bfloat16)
    Cin = None
    if c.beta != 0.0:
        gen.manual_seed(int(c.seed) + 1)
        Cin = _uniform((c.N, c.P, c.Q, c.K), gen, dev)
    return X, F, Cin


def conv_resolution(count: int = 64) -> List[Conv]:
    """The dynamic-resolution workload's layers as convolutions: the same draws
    (batch uniform on [1, 32], side uniform on [160, 320], stage s in 0..3),
    each a 3x3 stride-1 'same' convolution on an H x H input, H = ceil(side /
    (4 * 2^s)), C = K = 64 * 2^s.  Its GEMM is the dynamic-resolution GEMM."""
    rng = np.random.default_rng(1002)
    out = []
    for i in range(count):
        batch = int(rng.integers(1, 33))
        side = int(rng.integers(160, 321))
        s = int(rng.integers(0, 4))
        ch = 64 * 2 ** s
        h = math.ceil(side / (4 * 2 ** s))
        out.append(Conv(batch, h, h, ch, ch, seed=1000 + 800 + 7 * i))
    return out


CONV_WORKLOADS = {"conv_resolution": conv_resolution}


def grouped_experts(count: int = 48) -> List[Gemm]:
    """Non-uniform merged problems: 48 expert GEMMs of one layer, tokens per
    expert uniform on [1, 512], (N, K) = (2048, 1024).  BladeDISC's merge of
    same-shape GEMMs into a batched GEMM does not apply (every M differs); a
    grouped GEMM runs them in one launch."""
    rng = np.random.default_rng(1000 + 900)
    return [Gemm(int(rng.integers(1, 513)), 2048, 1024, seed=1000 + 900 + 7 * i) for i in range(count)]


GROUPED_WORKLOADS = {"grouped_experts": grouped_experts}


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a CPU tensor as numpy uint16 (no conversion)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# The five workloads.  seed = 1000 + workload index; problem i of a list uses
# seed = 1000 + 100 * index + 7 * i for its operands.
# ---------------------------------------------------------------------------

def single_skinny() -> List[Gemm]:
    """(105, 1024, 12544): the shape the MikPoly summary quotes a vendor GEMM on
    (Introduction, vendor-library table), alpha = beta = 1 with C uniform."""
    return [Gemm(105, 1024, 12544, alpha=1.0, beta=1.0, seed=1000)]


SEQ_NK = [(2304, 768), (768, 768), (3072, 768), (768, 3072)]


def dynamic_sequence(count: int = 64) -> List[Gemm]:
    """Dynamic sequence length (MikPoly summary, section 2 scenarios): M =
    8 * seq with seq uniform on [1, 512] per call; (N, K) cycles over a
    Transformer layer's four projections; beta = 0."""
    rng = np.random.default_rng(1001)
    seqs = rng.integers(1, 513, size=count)
    out = []
    for i, s in enumerate(seqs):
        N, K = SEQ_NK[i % len(SEQ_NK)]
        out.append(Gemm(int(8 * s), N, K, seed=1000 + 100 + 7 * i))
    return out


def dynamic_resolution(count: int = 64) -> List[Gemm]:
    """Dynamic image resolution, convolution lowered to GEMM (MikPoly summary,
    section 5: convolutions run as GEMM).  Batch uniform on [1, 32], square
    side uniform on [160, 320], one of four ResNet-50-like 3x3 stages s with
    Cin = Cout = 64 * 2^s:  N = Cout, K = 9 * Cin, H_out = ceil(side / (4 *
    2^s)), M = batch * H_out^2.  A is drawn directly as the im2col matrix."""
    rng = np.random.default_rng(1002)
    out = []
    for i in range(count):
        batch = int(rng.integers(1, 33))
        side = int(rng.integers(160, 321))
        s = int(rng.integers(0, 4))
        N = 64 * 2 ** s
        K = 9 * N
        h = math.ceil(side / (4 * 2 ** s))
        out.append(Gemm(batch * h * h, N, K, seed=1000 + 200 + 7 * i))
    return out


def merged_qkv(count: int = 64) -> List[Gemm]:
    """Shared-operand merge A x concat(Wq, Wk, Wv) (BladeDISC v0.2.0 notes,
    "GEMM merge" 1): K = 1024, N = 3 * 1024, M uniform on [1, 4096]."""
    rng = np.random.default_rng(1003)
    return [Gemm(int(m), 3072, 1024, seed=1000 + 300 + 7 * i)
            for i, m in enumerate(rng.integers(1, 4097, size=count))]


def merged_batched(count: int = 64) -> List[Gemm]:
    """Same-shape merge into one batched GEMM (BladeDISC v0.2.0 notes, "GEMM
    merge" 2): 12 problems of (seq, seq, 64), seq uniform on [16, 512]."""
    rng = np.random.default_rng(1004)
    return [Gemm(int(s), int(s), 64, batch=12, seed=1000 + 400 + 7 * i)
            for i, s in enumerate(rng.integers(16, 513, size=count))]


def stress(count: int = 1000) -> List[Gemm]:
    """Stress sweep: M, N, K each floor(exp(U[0, ln 16384])) clipped to
    [1, 16384], plus 4096^3; alpha = 1.5, beta = 0.5, C uniform."""
    rng = np.random.default_rng(1005)
    dims = np.floor(np.exp(rng.uniform(0.0, math.log(16384.0), size=(count, 3)))).astype(np.int64)
    dims = np.clip(dims, 1, 16384)
    out = [Gemm(int(m), int(n), int(k), alpha=1.5, beta=0.5, seed=1000 + 500 + 7 * i)
           for i, (m, n, k) in enumerate(dims)]
    out.append(Gemm(4096, 4096, 4096, alpha=1.5, beta=0.5, seed=1000 + 500 + 7 * count))
    return out


def b2b_adapter(count: int = 64) -> List[B2B]:
    """Bottleneck pairs at dynamic sequence length: M = 8 * seq (seq uniform
    in [1, 512], as in the dynamic-sequence workload), 768 -> 256 (ReLU) ->
    768.  N0 = 256 is the widest D0 one CTA keeps on chip."""
    rng = np.random.default_rng(1000 + 600)
    return [B2B(8 * int(rng.integers(1, 513)), 256, 768, 768, act0=1, seed=1000 + 600 + 7 * i)
            for i in range(count)]


def b2b_1x1(count: int = 64) -> List[B2B]:
    """Two consecutive 1x1 convolutions as GEMMs at dynamic resolution (the
    BOLT summary's deepening with 1x1 convolutions): M = batch * H * W with
    batch in [1, 32] and H = W in {7, 14, 28, 56}, channels 256 -> 64 (ReLU)
    -> 256."""
    rng = np.random.default_rng(1000 + 700)
    out = []
    for i in range(count):
        batch = int(rng.integers(1, 33))
        hw = int(rng.choice([7, 14, 28, 56]))
        out.append(B2B(batch * hw * hw, 64, 256, 256, act0=1, seed=1000 + 700 + 7 * i))
    return out


B2B_WORKLOADS = {"b2b_adapter": b2b_adapter, "b2b_1x1": b2b_1x1}


WORKLOADS = {
    "single_skinny": single_skinny,
    "dynamic_sequence": dynamic_sequence,
    "dynamic_resolution": dynamic_resolution,
    "merged_qkv": merged_qkv,
    "merged_batched": merged_batched,
    "stress": stress,
}


def workload(name: str, count: Optional[int] = None) -> List[Gemm]:
    fn = WORKLOADS[name]
    return fn() if count is None or name == "single_skinny" else fn(count)

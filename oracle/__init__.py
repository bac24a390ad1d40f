"""fp64 CPU oracle for D = alpha*A*B + beta*C -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` leg of
``bench.py`` may import this package.  The GPU library never loads it and
shares no code with it: the arithmetic lives in ``mp_oracle.c`` (plain C,
fp64, no fused multiply-add), and this module only marshals numpy arrays.

Operands: A and B are bf16 bit patterns (numpy ``uint16``), row-major with
leading dimensions; C is ``float32`` (ignored when beta == 0).  Every result is
``float64``.

What each routine follows (page titles and sections):
  * ``gemm_naive``  -- MikPoly summary, preliminaries part 2 (loop tiling structure): the plain i-j-k nest,
    then the BOLT summary's epilogue ``alpha*A*W + beta*C``.
  * ``gemm_tiled``  -- MikPoly summary, preliminaries part 2 (loop tiling structure): the TILE_SIZE 32 nest
    (zeroed output, edges clamped).
  * ``gemm_rows``   -- the same definition in i-k-j order over OpenMP rows.
  * ``gemm_entries`` / ``magnitude`` / ``freivalds`` -- the same definition
    evaluated at chosen entries, its element-wise magnitude, and a
    matrix-vector probe for outputs too large to recompute.
  * ``epilogue`` -- the activation of the epilogue variants, applied in fp64
    to alpha*A*B + beta*C: ReLU max(x, 0), GELU x*Phi(x) with Phi the standard
    normal distribution function (BOLT summary, "Persistent kernel (GEMM/Conv)
    fusion": activations as further epilogue stages).
  * ``bf16_round`` -- fp64 values rounded to bf16 (nearest even), for the
    bf16-output variant; ``within_bound_out`` the parity bound with the
    activation's slope and one bf16 unit of the reference added.
  * ``b2b`` -- back-to-back GEMMs (BOLT summary, "Persistent kernel
    (GEMM/Conv) fusion"): D0 = alpha0*A0*W0 + beta0*C0, then
    D1 = alpha1*D0*W1 + beta1*C1, in fp64 with no rounding of D0; an optional
    activation on D0 (the epilogue variants above) sits between the two.
    ``b2b_bound`` carries the stated per-GEMM bound through the second GEMM
    and adds one bf16 rounding of D0 (the operand type of the second GEMM
    when D0 stays on chip).
  * ``conv2d_nhwc`` -- a stride-1 2-D convolution (MikPoly summary, section 5:
    convolutions run as GEMM), written as its definition: for every filter
    tap (r, s), the zero-padded input shifted by (r, s) times that tap's
    C x K slice, summed over taps; then alpha and beta*Cin as for a GEMM.
    ``conv2d_magnitude`` is the same sum over absolute values (the
    tolerance scale, as ``magnitude`` for a GEMM); ``im2col_nhwc`` builds the
    explicit [N*P*Q, R*S*C] matrix that a GEMM-based convolution multiplies.
  * ``gemm_group`` -- a group of independent GEMMs of different shapes
    (BladeDISC v0.2.0 notes, GEMM merging, widened from same-shape problems
    to any shapes): the definition applied to each problem.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mp_oracle.c")
_LIB = os.path.join(_HERE, "libmp_oracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_dbl = ctypes.c_double
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile mp_oracle.c into libmp_oracle.so with gcc (OpenMP, fp-contract off)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            gemm_args = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _dbl, _dbl, _vp, _i64]
            for name in ("oracle_gemm_naive", "oracle_gemm_tiled"):
                f = getattr(lib, name)
                f.argtypes = gemm_args
                f.restype = None
            lib.oracle_gemm_rows.argtypes = gemm_args + [ctypes.c_int]
            lib.oracle_gemm_rows.restype = ctypes.c_int
            lib.oracle_gemm_entries.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64,
                                                _dbl, _dbl, _i64, _vp, _vp, _vp, _vp]
            lib.oracle_gemm_entries.restype = None
            lib.oracle_gemm_magnitude.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp,
                                                  _i64, _dbl, _vp, _i64]
            lib.oracle_gemm_magnitude.restype = None
            lib.oracle_freivalds.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64,
                                             _dbl, _dbl, _vp, _i64, _vp, _vp, _vp, _vp, _vp]
            lib.oracle_freivalds.restype = None
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _operands(A, B, C, beta):
    A = np.ascontiguousarray(A, dtype=np.uint16) if A.dtype != np.uint16 else A
    B = np.ascontiguousarray(B, dtype=np.uint16) if B.dtype != np.uint16 else B
    if beta != 0.0:
        if C is None:
            raise ValueError("beta != 0 needs C")
        if C.dtype != np.float32:
            raise TypeError("C must be float32")
    else:
        C = None
    for X in (A, B) + ((C,) if C is not None else ()):
        if X.ndim != 2 or (X.size and X.shape[1] > 1 and X.strides[1] != X.itemsize):
            raise ValueError("operands must be 2-D with unit column stride")
    return A, B, C


def _ld(X):
    if X is None:
        return 0
    if X.size == 0 or X.shape[0] == 1:
        return max(1, X.shape[1])
    return X.strides[0] // X.itemsize


def _shape(A, B):
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner sizes differ: A is {A.shape}, B is {B.shape}")
    return M, N, K


def _gemm(name, A, B, C, alpha, beta, threads=None):
    lib = _load()
    A, B, C = _operands(A, B, C, beta)
    M, N, K = _shape(A, B)
    D = np.empty((M, N), dtype=np.float64)
    args = [M, N, K, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C),
            float(alpha), float(beta), _ptr(D), N]
    if threads is None:
        getattr(lib, name)(*args)
        return D
    used = lib.oracle_gemm_rows(*args, int(threads))
    return D, used


def gemm_naive(A, B, C=None, alpha=1.0, beta=0.0) -> np.ndarray:
    """Plain i-j-k nest (MikPoly summary, preliminaries part 2) with the alpha/beta epilogue."""
    return _gemm("oracle_gemm_naive", A, B, C, alpha, beta)


def gemm_tiled(A, B, C=None, alpha=1.0, beta=0.0) -> np.ndarray:
    """Loop-tiled nest, TILE_SIZE 32 (MikPoly summary, preliminaries part 2), edges clamped."""
    return _gemm("oracle_gemm_tiled", A, B, C, alpha, beta)


def gemm_rows(A, B, C=None, alpha=1.0, beta=0.0, threads: int = 0):
    """Same definition, i-k-j order, OpenMP over rows.  Returns (D, threads_used)."""
    return _gemm("oracle_gemm_rows", A, B, C, alpha, beta, threads=threads)


def gemm(A, B, C=None, alpha=1.0, beta=0.0) -> np.ndarray:
    """The oracle's default full evaluation (row-parallel)."""
    return gemm_rows(A, B, C, alpha, beta)[0]


def gemm_entries(A, B, C, alpha, beta, rows, cols):
    """Entries (rows[t], cols[t]) of the definition and their magnitudes."""
    lib = _load()
    A, B, C = _operands(A, B, C, beta)
    M, N, K = _shape(A, B)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows and cols differ in length")
    if rows.size and (rows.min() < 0 or rows.max() >= M or cols.min() < 0 or cols.max() >= N):
        raise IndexError("entry outside the output")
    out = np.empty(rows.size, dtype=np.float64)
    mag = np.empty(rows.size, dtype=np.float64)
    lib.oracle_gemm_entries(M, N, K, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C),
                            float(alpha), float(beta), rows.size, _ptr(rows), _ptr(cols),
                            _ptr(out), _ptr(mag))
    return out, mag


def magnitude(A, B, C=None, beta=0.0) -> np.ndarray:
    """sum_k |A_ik||B_kj| + |beta*C_ij| for every entry (the tolerance scale)."""
    lib = _load()
    A, B, C = _operands(A, B, C, beta)
    M, N, K = _shape(A, B)
    G = np.empty((M, N), dtype=np.float64)
    lib.oracle_gemm_magnitude(M, N, K, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C),
                              float(beta), _ptr(G), N)
    return G


def freivalds(A, B, C, alpha, beta, D, x):
    """Residual y = D x - (alpha A (B x) + beta C x) and its row magnitudes."""
    lib = _load()
    A, B, C = _operands(A, B, C, beta)
    M, N, K = _shape(A, B)
    D = np.ascontiguousarray(D, dtype=np.float32)
    if D.shape != (M, N):
        raise ValueError("D has the wrong shape")
    x = np.ascontiguousarray(x, dtype=np.float64)
    bx = np.empty(K, dtype=np.float64)
    abx = np.empty(K, dtype=np.float64)
    y = np.empty(M, dtype=np.float64)
    ymag = np.empty(M, dtype=np.float64)
    lib.oracle_freivalds(M, N, K, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C),
                         float(alpha), float(beta), _ptr(D), N, _ptr(x), _ptr(bx), _ptr(abx),
                         _ptr(y), _ptr(ymag))
    return y, ymag


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (high half of an fp32 word) to fp64."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# The parity bound stated for bf16 inputs with fp32 accumulation and fp32 output:
#   |D - D_ref| <= 2e-3 * (sum_k |A_ik||B_kj| + |beta*C_ij|)
PARITY_RTOL = 2e-3

ACT_NONE, ACT_RELU, ACT_GELU = 0, 1, 2
# Largest slope of the activations: ReLU 1; GELU x*Phi(x) has
# d/dx = Phi(x) + x*phi(x), largest near x = 1.414 (about 1.1289).
ACT_SLOPE = {ACT_NONE: 1.0, ACT_RELU: 1.0, ACT_GELU: 1.1290}


def epilogue(X, act: int) -> np.ndarray:
    """The activation of the epilogue variants, in fp64."""
    import math
    X = np.asarray(X, dtype=np.float64)
    if act == ACT_NONE:
        return X.copy()
    if act == ACT_RELU:
        return np.maximum(X, 0.0)
    if act == ACT_GELU:
        erf = np.vectorize(math.erf, otypes=[np.float64])
        return X * 0.5 * (1.0 + erf(X / math.sqrt(2.0)))
    raise ValueError(f"unknown activation {act}")


def bf16_round(X) -> np.ndarray:
    """fp64 -> nearest bf16 (ties to even), returned as fp64: the value rounded
    once to fp32 by the same rule, then its low 16 bits rounded off."""
    f = np.asarray(X, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32).astype(np.float64)
    return np.where(np.isnan(f), np.nan, out)


def within_bound_out(D, Dref_act, mag, act: int, bf16: bool, rtol: float = PARITY_RTOL):
    """Parity of an epilogue variant: |D - act(Dref)| <= rtol * slope(act) * mag
    (the stated bound carried through the activation), plus one bf16 unit of
    act(Dref) when D is bf16 (the output's own rounding)."""
    D = np.asarray(D, dtype=np.float64)
    bound = rtol * ACT_SLOPE[act] * np.asarray(mag, dtype=np.float64)
    if bf16:
        bound = bound + np.abs(Dref_act) * 2.0 ** -8
    err = np.abs(D - Dref_act)
    ok = bool(np.all(err <= bound))
    worst = float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0
    return ok, worst


def within_bound(D, Dref, mag, rtol: float = PARITY_RTOL):
    """Element-wise check of the parity bound; returns (ok, worst ratio)."""
    D = np.asarray(D, dtype=np.float64)
    err = np.abs(D - Dref)
    lim = rtol * mag
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(lim > 0, err / np.where(lim > 0, lim, 1.0), np.where(err > 0, np.inf, 0.0))
    ok = bool(np.all(np.isfinite(D)) and np.all(err <= lim))
    return ok, float(ratio.max()) if ratio.size else 0.0


def b2b(A0, W0, C0, W1, C1, alpha0, beta0, alpha1, beta1, act0: int = ACT_NONE):
    """D1 = alpha1 * act0(alpha0 A0 W0 + beta0 C0) W1 + beta1 C1 in fp64.

    A0 [M, K0], W0 [K0, N0] and W1 [N0, N1] are bf16 bit patterns; C0 [M, N0]
    and C1 [M, N1] float32 (ignored when their beta is 0).  Returns (D1, D0),
    D0 after the activation."""
    D0 = epilogue(gemm(A0, W0, C0, alpha0, beta0), act0)
    W1f = bf16_bits_to_f64(W1)
    if D0.shape[1] != W1f.shape[0]:
        raise ValueError("W1 rows must equal the columns of D0")
    D1 = alpha1 * (D0 @ W1f)
    if beta1 != 0.0:
        D1 = D1 + beta1 * np.asarray(C1, dtype=np.float64)
    return D1, D0


def b2b_bound(A0, W0, C0, W1, C1, alpha0, beta0, alpha1, beta1, act0, D0, rtol: float = PARITY_RTOL):
    """Element-wise bound on |D1 - D1_ref| for the fused back-to-back GEMM.

    The first GEMM is within e0 = rtol * (|alpha0| sum|A0||W0| + |beta0 C0|);
    the activation (slope at most L) carries it as L*e0; D0 is then rounded to
    bf16 (at most 2^-8 of its value); the second GEMM adds its own stated bound
    rtol * (|alpha1| |D0| |W1| + |beta1 C1|).  So
      bound = rtol*mag1 + |alpha1| * ((L e0 (1 + 2^-8) + 2^-8 |D0|) |W1|)."""
    u = 2.0 ** -8
    e0 = rtol * (abs(alpha0) * magnitude(A0, W0) +
                 (abs(beta0) * np.abs(np.asarray(C0, dtype=np.float64)) if beta0 != 0.0 else 0.0))
    absW1 = np.abs(bf16_bits_to_f64(W1))
    absD0 = np.abs(np.asarray(D0, dtype=np.float64))
    mag1 = abs(alpha1) * (absD0 @ absW1)
    if beta1 != 0.0:
        mag1 = mag1 + abs(beta1) * np.abs(np.asarray(C1, dtype=np.float64))
    carried = abs(alpha1) * ((ACT_SLOPE[act0] * e0 * (1.0 + u) + u * absD0) @ absW1)
    return rtol * mag1 + carried


def within_b2b(D1, D1ref, bound):
    """(every |D1 - D1ref| <= bound and D1 finite, worst err/bound)."""
    D1 = np.asarray(D1, dtype=np.float64)
    err = np.abs(D1 - D1ref)
    ok = bool(np.all(np.isfinite(D1)) and np.all(err <= bound))
    worst = float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0
    return ok, worst


def _conv_out(H, W, R, S, pad_h, pad_w):
    return H + 2 * pad_h - R + 1, W + 2 * pad_w - S + 1


def _conv_taps(Xf, Wf, pad_h, pad_w):
    """sum over taps (r, s) of the shifted, zero-padded input times Wf[r, s]."""
    N, H, W, C = Xf.shape
    R, S, C2, K = Wf.shape
    if C2 != C:
        raise ValueError("filter channels must match the input's")
    P, Q = _conv_out(H, W, R, S, pad_h, pad_w)
    Xp = np.zeros((N, H + 2 * pad_h, W + 2 * pad_w, C), dtype=np.float64)
    Xp[:, pad_h:pad_h + H, pad_w:pad_w + W, :] = Xf
    D = np.zeros((N, P, Q, K), dtype=np.float64)
    for r in range(R):
        for s in range(S):
            D += Xp[:, r:r + P, s:s + Q, :] @ Wf[r, s]
    return D


def conv2d_nhwc(X, Wt, Cin=None, alpha=1.0, beta=0.0, pad_h=1, pad_w=1):
    """D[n,p,q,k] = alpha * sum_{r,s,c} X[n, p+r-pad_h, q+s-pad_w, c] * Wt[r,s,c,k]
    + beta * Cin[n,p,q,k]  (stride 1, zero padding), in fp64.

    X [N,H,W,C] and Wt [R,S,C,K] are bf16 bit patterns; Cin [N,P,Q,K] float32
    (ignored when beta == 0)."""
    D = alpha * _conv_taps(bf16_bits_to_f64(X), bf16_bits_to_f64(Wt), pad_h, pad_w)
    if beta != 0.0:
        D = D + beta * np.asarray(Cin, dtype=np.float64)
    return D


def conv2d_magnitude(X, Wt, Cin=None, beta=0.0, pad_h=1, pad_w=1):
    """sum_{r,s,c} |X||Wt| + |beta*Cin| at every output (the tolerance scale)."""
    G = _conv_taps(np.abs(bf16_bits_to_f64(X)), np.abs(bf16_bits_to_f64(Wt)), pad_h, pad_w)
    if beta != 0.0:
        G = G + abs(beta) * np.abs(np.asarray(Cin, dtype=np.float64))
    return G


def im2col_nhwc(X, R, S, pad_h=1, pad_w=1):
    """The [N*P*Q, R*S*C] matrix of a GEMM-based convolution: row (n, p, q),
    column (r, s, c) holds X[n, p+r-pad_h, q+s-pad_w, c] (0 outside the input).
    Returns bf16 bit patterns (a copy of X's bits, zeros as 0x0000)."""
    X = np.asarray(X, dtype=np.uint16)
    N, H, W, C = X.shape
    P, Q = _conv_out(H, W, R, S, pad_h, pad_w)
    out = np.zeros((N, P, Q, R, S, C), dtype=np.uint16)
    for r in range(R):
        for s in range(S):
            for p in range(P):
                h = p + r - pad_h
                if not 0 <= h < H:
                    continue
                for q in range(Q):
                    w = q + s - pad_w
                    if 0 <= w < W:
                        out[:, p, q, r, s, :] = X[:, h, w, :]
    return out.reshape(N * P * Q, R * S * C)


def gemm_group(problems):
    """[(D_i, magnitude_i)] for problems given as (A_bits, B_bits, C, alpha,
    beta) tuples: each problem's own definition, nothing shared."""
    return [(gemm(A, B, C, alpha, beta), magnitude(A, B, C, beta)) for (A, B, C, alpha, beta) in problems]

"""Python binding of the mp C ABI (dynamic-shape GEMM D = alpha*A*B + beta*C on GB300).

Argument marshalling only: every function here forwards to the entry point of
the same name in ``libmp.so`` (declared in ``include/mp.h``); the planning and
every step of the GEMM run in that library and its CUDA kernels.  Torch
tensors supply device memory and streams.  A missing or unloadable library is
an error -- there is no other code path.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

from . import _build

__all__ = [
    "MPError", "mp_init", "mp_init_host", "mp_destroy", "mp_plan", "mp_plan_batched", "mp_plan_many",
    "mp_evaluate_plan", "mp_gemm", "mp_gemm_batched", "mp_check", "mp_force_plan", "mp_get_hw",
    "mp_set_kernel_model", "mp_set_split_model", "mp_get_split_model", "mp_load_calibration", "mp_inject_wait_timeout", "mp_status_string", "library", "mp_gemm_noalloc",
    "mp_check_noalloc", "mp_noalloc_inject_wait_timeout",
    "mp_enumerate_plans", "mp_gemm_with_plan", "mp_set_plan_mode", "MP_PLAN_MIKPOLY", "MP_PLAN_WAVE",
    "MP_PLAN_PIPE", "mp_gemm_ex", "MP_ACT_NONE", "MP_ACT_RELU", "MP_ACT_GELU", "MP_EPI_OUT_BF16",
    "MpHw", "MpKernelDesc", "MpRegionInfo", "MpPlanInfo", "MP_MAX_REGIONS", "MP_MAX_KERNELS",
    "mp_gemm_b2b", "mp_plan_b2b", "MpB2BPlan", "mp_set_b2b_mode", "MP_B2B_AUTO", "MP_B2B_FUSED",
    "MP_B2B_TWO_LAUNCH", "mp_conv2d", "mp_plan_conv", "MpConvPlan",
    "mp_gemm_grouped", "mp_plan_grouped", "MpGemmProblem", "MpGroupedPlan",
]

MP_MAX_REGIONS = 4
MP_MAX_KERNELS = 16

MP_ACT_NONE = 0
MP_ACT_RELU = 1
MP_ACT_GELU = 2
MP_EPI_OUT_BF16 = 0x100

MP_PLAN_MIKPOLY = 0
MP_PLAN_WAVE = 1
MP_PLAN_PIPE = 2

MP_OK = 0
MP_ERR_INVALID_ARG = -1
MP_ERR_UNSUPPORTED = -2
MP_ERR_CUDA = -3
MP_ERR_PLAN = -4
MP_ERR_DEVICE_TIMEOUT = -5
MP_ERR_NO_MEMORY = -6


class MpHw(ctypes.Structure):
    _fields_ = [("num_pe", ctypes.c_int32), ("warps_per_wave", ctypes.c_int32),
                ("local_mem_bytes", ctypes.c_int64), ("shared_mem_bytes", ctypes.c_int64),
                ("hbm_gbs", ctypes.c_double), ("l2_gbs", ctypes.c_double),
                ("mma_tflops", ctypes.c_double)]


class MpKernelDesc(ctypes.Structure):
    _fields_ = [("um", ctypes.c_int32), ("un", ctypes.c_int32), ("uk", ctypes.c_int32),
                ("warps", ctypes.c_int32), ("swap", ctypes.c_int32), ("pair", ctypes.c_int32),
                ("fixed_us", ctypes.c_double), ("per_step_us", ctypes.c_double), ("tail_us", ctypes.c_double)]


class MpRegionInfo(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("um", ctypes.c_int32), ("un", ctypes.c_int32),
                ("uk", ctypes.c_int32), ("swap", ctypes.c_int32), ("pair", ctypes.c_int32),
                ("m0", ctypes.c_int64), ("n0", ctypes.c_int64),
                ("m_ext", ctypes.c_int64), ("n_ext", ctypes.c_int64),
                ("splits", ctypes.c_int32), ("f_num", ctypes.c_int32),
                ("f_parallel", ctypes.c_int64), ("f_wave", ctypes.c_int64),
                ("f_pipe_us", ctypes.c_double)]


class MpPlanInfo(ctypes.Structure):
    _fields_ = [("pattern", ctypes.c_int32), ("num_regions", ctypes.c_int32),
                ("region", MpRegionInfo * MP_MAX_REGIONS), ("cost_us", ctypes.c_double),
                ("total_tasks", ctypes.c_int64), ("evaluated", ctypes.c_int32),
                ("pruned", ctypes.c_int32), ("workspace_bytes", ctypes.c_int64)]

    def regions(self):
        return [self.region[i] for i in range(self.num_regions)]


class MpB2BPlan(ctypes.Structure):
    _fields_ = [("n0p", ctypes.c_int32), ("bn1", ctypes.c_int32), ("chunks", ctypes.c_int32),
                ("mblocks", ctypes.c_int32), ("cpg", ctypes.c_int32), ("units", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("num_stages", ctypes.c_int32), ("stage_bytes", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("cost_us", ctypes.c_double), ("mode", ctypes.c_int32),
                ("two_launch_cost_us", ctypes.c_double)]


class MpConvPlan(ctypes.Structure):
    _fields_ = [("wb", ctypes.c_int32), ("hb", ctypes.c_int32), ("nb", ctypes.c_int32), ("bn", ctypes.c_int32),
                ("tiles_q", ctypes.c_int32), ("tiles_p", ctypes.c_int32), ("tiles_n", ctypes.c_int32),
                ("tiles_k", ctypes.c_int32), ("ksteps", ctypes.c_int32), ("tiles", ctypes.c_int32),
                ("splits", ctypes.c_int32), ("units", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("num_stages", ctypes.c_int32), ("stage_bytes", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("useful", ctypes.c_double), ("cost_us", ctypes.c_double)]


class MpGemmProblem(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("A", ctypes.c_void_p), ("lda", ctypes.c_int64), ("B", ctypes.c_void_p), ("ldb", ctypes.c_int64),
                ("C", ctypes.c_void_p), ("ldc", ctypes.c_int64), ("D", ctypes.c_void_p), ("ldd", ctypes.c_int64),
                ("alpha", ctypes.c_float), ("beta", ctypes.c_float)]


class MpGroupedPlan(ctypes.Structure):
    _fields_ = [("bn", ctypes.c_int32), ("units", ctypes.c_int32), ("launches", ctypes.c_int32),
                ("num_stages", ctypes.c_int32), ("stage_bytes", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("cost_us", ctypes.c_double)]


class MPError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {mp_status_string(status)} ({status})")


_lock = threading.Lock()
_lib = None
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_vp = ctypes.c_void_p
_f = ctypes.c_float


def library(build: bool = True) -> ctypes.CDLL:
    """Load libmp.so (building it in-tree first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build:
                path = _build.build()
            if not os.path.exists(path):
                raise OSError(f"libmp.so not built at {path}")
            lib = ctypes.CDLL(path)
            sig = {
                "mp_init": ([ctypes.POINTER(_vp), ctypes.c_int, ctypes.c_char_p], ctypes.c_int),
                "mp_init_host": ([ctypes.POINTER(_vp), ctypes.POINTER(MpHw), ctypes.POINTER(MpKernelDesc),
                                  _i32], ctypes.c_int),
                "mp_destroy": ([_vp], ctypes.c_int),
                "mp_plan": ([_vp, _i64, _i64, _i64, ctypes.POINTER(MpPlanInfo)], ctypes.c_int),
                "mp_plan_batched": ([_vp, _i64, _i64, _i64, _i64, ctypes.POINTER(MpPlanInfo)], ctypes.c_int),
                "mp_plan_many": ([_vp, _i32, ctypes.POINTER(_i64), ctypes.POINTER(MpPlanInfo)], ctypes.c_int),
                "mp_evaluate_plan": ([_vp, _i64, _i64, _i64, _i64, ctypes.POINTER(MpPlanInfo)], ctypes.c_int),
                "mp_gemm": ([_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64,
                             _f, _f, _vp], ctypes.c_int),
                "mp_gemm_batched": ([_vp, _i64, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _i64,
                                     _vp, _i64, _i64, _vp, _i64, _i64, _f, _f, _vp], ctypes.c_int),
                "mp_gemm_noalloc": ([_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64,
                                     _f, _f, _vp], ctypes.c_int),
                "mp_check": ([_vp, _vp], ctypes.c_int),
                "mp_check_noalloc": ([_vp], ctypes.c_int),
                "mp_noalloc_inject_wait_timeout": ([_i32, _i64], ctypes.c_int),
                "mp_force_plan": ([_vp, _i32, _i32], ctypes.c_int),
                "mp_get_hw": ([_vp, ctypes.POINTER(MpHw), ctypes.POINTER(MpKernelDesc),
                               ctypes.POINTER(_i32)], ctypes.c_int),
                "mp_set_kernel_model": ([_vp, _i32, ctypes.c_double, ctypes.c_double, ctypes.c_double], ctypes.c_int),
                "mp_set_split_model": ([_vp, _i32, _i32, ctypes.c_double, ctypes.c_double], ctypes.c_int),
                "mp_load_calibration": ([_vp, ctypes.c_char_p], ctypes.c_int),
                "mp_get_split_model": ([_vp, _i32, _i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)],
                                       ctypes.c_int),
                "mp_inject_wait_timeout": ([_vp, _i32, _i64], ctypes.c_int),
                "mp_status_string": ([ctypes.c_int], ctypes.c_char_p),
                "mp_enumerate_plans": ([_vp, _i64, _i64, _i64, _i64, ctypes.POINTER(MpPlanInfo), _i32,
                                        ctypes.POINTER(_i32)], ctypes.c_int),
                "mp_gemm_with_plan": ([_vp, ctypes.POINTER(MpPlanInfo), _i64, _i64, _i64, _vp, _i64, _vp, _i64,
                                       _vp, _i64, _vp, _i64, _f, _f, _vp], ctypes.c_int),
                "mp_set_plan_mode": ([_vp, _i32], ctypes.c_int),
                "mp_gemm_ex": ([_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64,
                                _f, _f, _i32, _vp], ctypes.c_int),
                "mp_gemm_b2b": ([_vp, _i64, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64,
                                 _vp, _i64, _vp, _i64, _f, _f, _f, _f, _i32, _vp], ctypes.c_int),
                "mp_plan_b2b": ([_vp, _i64, _i64, _i64, _i64, ctypes.POINTER(MpB2BPlan)], ctypes.c_int),
                "mp_set_b2b_mode": ([_vp, _i32], ctypes.c_int),
                "mp_gemm_grouped": ([_vp, _i32, ctypes.POINTER(MpGemmProblem), _vp], ctypes.c_int),
                "mp_plan_grouped": ([_vp, _i32, ctypes.POINTER(MpGemmProblem), ctypes.POINTER(MpGroupedPlan)],
                                    ctypes.c_int),
                "mp_conv2d": ([_vp, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _i64,
                               _vp, _i64, _f, _f, _vp], ctypes.c_int),
                "mp_plan_conv": ([_vp, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64,
                                  ctypes.POINTER(MpConvPlan)], ctypes.c_int),
            }
            for name, (args, res) in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def mp_status_string(status: int) -> str:
    return library().mp_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != MP_OK:
        raise MPError(status, where)


class Handle:
    """Owns one mp_handle; destroyed with mp_destroy when closed or collected."""

    def __init__(self, ptr: int, device: Optional[int]):
        self.ptr = ptr
        self.device = device

    def close(self) -> None:
        if self.ptr:
            library().mp_destroy(self.ptr)
            self.ptr = None

    def __del__(self):  # pragma: no cover - best effort at interpreter exit
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def mp_init(device: int = 0, calib_path: Optional[str] = None) -> Handle:
    """calib_path None: the measured GB300 table shipped in calib/gb300.txt;
    "": the analytic model; otherwise the table at that path."""
    out = _vp()
    _check(library().mp_init(ctypes.byref(out), int(device),
                             os.fsencode(calib_path) if calib_path is not None else None), "mp_init")
    return Handle(out.value, device)


def mp_init_host(hw: MpHw, kernels=None) -> Handle:
    out = _vp()
    if kernels:
        arr = (MpKernelDesc * len(kernels))(*kernels)
        st = library().mp_init_host(ctypes.byref(out), ctypes.byref(hw), arr, len(kernels))
    else:
        st = library().mp_init_host(ctypes.byref(out), ctypes.byref(hw), None, 0)
    _check(st, "mp_init_host")
    return Handle(out.value, None)


def mp_destroy(h: Handle) -> None:
    h.close()


def mp_plan(h: Handle, M: int, N: int, K: int) -> MpPlanInfo:
    info = MpPlanInfo()
    _check(library().mp_plan(h.ptr, M, N, K, ctypes.byref(info)), "mp_plan")
    return info


def mp_plan_batched(h: Handle, batch: int, M: int, N: int, K: int) -> MpPlanInfo:
    info = MpPlanInfo()
    _check(library().mp_plan_batched(h.ptr, batch, M, N, K, ctypes.byref(info)), "mp_plan_batched")
    return info


def mp_plan_many(h: Handle, shapes, want_plans: bool = True):
    """Plan a list of (M, N, K) in one library call; returns the plans (or
    None when want_plans is False, which only runs the searches)."""
    n = len(shapes)
    flat = (_i64 * (3 * n))(*[int(x) for s in shapes for x in s])
    out = (MpPlanInfo * max(1, n))() if want_plans else None
    _check(library().mp_plan_many(h.ptr, n, flat, out), "mp_plan_many")
    return [out[i] for i in range(n)] if want_plans else None


def mp_evaluate_plan(h: Handle, batch: int, M: int, N: int, K: int, regions) -> MpPlanInfo:
    """regions: list of dicts with kernel, m0, n0, m_ext, n_ext, splits."""
    info = MpPlanInfo()
    info.num_regions = len(regions)
    for i, r in enumerate(regions):
        g = info.region[i]
        g.kernel, g.m0, g.n0 = r["kernel"], r["m0"], r["n0"]
        g.m_ext, g.n_ext, g.splits = r["m_ext"], r["n_ext"], r.get("splits", 1)
    _check(library().mp_evaluate_plan(h.ptr, batch, M, N, K, ctypes.byref(info)), "mp_evaluate_plan")
    return info


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return int(getattr(stream, "cuda_stream", stream))


def _ld(t, name: str) -> int:
    if t.dim() < 2:
        raise ValueError(f"{name} must have at least 2 dimensions")
    if t.size(-1) > 1 and t.stride(-1) != 1:
        raise ValueError(f"{name} must have unit stride along its last dimension")
    return t.stride(-2) if t.size(-2) > 1 else max(1, t.size(-1))


def mp_gemm(h: Handle, A, B, C, D, alpha: float = 1.0, beta: float = 0.0, stream=None) -> None:
    """D = alpha*A@B + beta*C with torch CUDA tensors (A, B bf16; C, D fp32)."""
    import torch
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16 or D.dtype != torch.float32:
        raise TypeError("A and B must be bfloat16, D float32")
    M, K = A.shape[-2], A.shape[-1]
    N = B.shape[-1]
    if B.shape[-2] != K or D.shape[-2:] != (M, N):
        raise ValueError("shape mismatch")
    c_ptr, ldc = None, 0
    if beta != 0.0:
        if C is None or C.dtype != torch.float32 or C.shape[-2:] != (M, N):
            raise ValueError("beta != 0 needs an fp32 C of D's shape")
        c_ptr, ldc = C.data_ptr(), _ld(C, "C")
    st = library().mp_gemm(h.ptr, M, N, K, A.data_ptr(), _ld(A, "A"), B.data_ptr(), _ld(B, "B"),
                           c_ptr, ldc, D.data_ptr(), _ld(D, "D"), float(alpha), float(beta),
                           _stream_ptr(stream))
    _check(st, "mp_gemm")


def _gemm_args(A, B, C, D, beta, d_types=("float32",)):
    import torch
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16 or str(D.dtype).split(".")[-1] not in d_types:
        raise TypeError(f"A and B must be bfloat16, D one of {d_types}")
    M, K = A.shape[-2], A.shape[-1]
    N = B.shape[-1]
    if B.shape[-2] != K or D.shape[-2:] != (M, N):
        raise ValueError("shape mismatch")
    c_ptr, ldc = None, 0
    if beta != 0.0:
        if C is None or C.dtype != torch.float32 or C.shape[-2:] != (M, N):
            raise ValueError("beta != 0 needs an fp32 C of D's shape")
        c_ptr, ldc = C.data_ptr(), _ld(C, "C")
    return M, N, K, c_ptr, ldc


def mp_gemm_with_plan(h: Handle, plan: MpPlanInfo, A, B, C, D, alpha: float = 1.0, beta: float = 0.0,
                      stream=None) -> None:
    """mp_gemm with an explicit plan (from mp_plan, mp_enumerate_plans, or built by hand)."""
    M, N, K, c_ptr, ldc = _gemm_args(A, B, C, D, beta)
    st = library().mp_gemm_with_plan(h.ptr, ctypes.byref(plan), M, N, K, A.data_ptr(), _ld(A, "A"), B.data_ptr(),
                                     _ld(B, "B"), c_ptr, ldc, D.data_ptr(), _ld(D, "D"), float(alpha), float(beta),
                                     _stream_ptr(stream))
    _check(st, "mp_gemm_with_plan")


def mp_gemm_ex(h: Handle, A, B, C, D, alpha: float = 1.0, beta: float = 0.0, act: int = MP_ACT_NONE,
               stream=None) -> None:
    """D = act(alpha*A@B + beta*C); D float32 or bfloat16 (the output bit of
    the epilogue word follows D's dtype); C float32."""
    import torch
    M, N, K, c_ptr, ldc = _gemm_args(A, B, C, D, beta, d_types=("float32", "bfloat16"))
    epi = int(act) | (MP_EPI_OUT_BF16 if D.dtype == torch.bfloat16 else 0)
    st = library().mp_gemm_ex(h.ptr, M, N, K, A.data_ptr(), _ld(A, "A"), B.data_ptr(), _ld(B, "B"), c_ptr, ldc,
                              D.data_ptr(), _ld(D, "D"), float(alpha), float(beta), epi, _stream_ptr(stream))
    _check(st, "mp_gemm_ex")


def mp_gemm_b2b(h: Handle, A0, W0, C0, W1, C1, D1, alpha0: float = 1.0, beta0: float = 0.0, alpha1: float = 1.0,
                beta1: float = 0.0, act0: int = MP_ACT_NONE, stream=None) -> None:
    """D1 = alpha1 * act0(alpha0*A0@W0 + beta0*C0) @ W1 + beta1*C1 in one launch,
    the intermediate kept on chip (A0, W0, W1 bf16; C0, C1, D1 float32)."""
    import torch
    for name, t in (("A0", A0), ("W0", W0), ("W1", W1)):
        if t.dtype != torch.bfloat16 or t.dim() != 2:
            raise TypeError(f"{name} must be a 2-D bfloat16 tensor")
    if D1.dtype != torch.float32 or D1.dim() != 2:
        raise TypeError("D1 must be a 2-D float32 tensor")
    M, K0 = A0.shape
    N0 = W0.shape[1]
    N1 = W1.shape[1]
    if W0.shape[0] != K0 or W1.shape[0] != N0 or tuple(D1.shape) != (M, N1):
        raise ValueError("shape mismatch")
    c0, ldc0, c1, ldc1 = None, 0, None, 0
    if beta0 != 0.0:
        if C0 is None or C0.dtype != torch.float32 or tuple(C0.shape) != (M, N0):
            raise ValueError("beta0 != 0 needs an fp32 C0 of shape (M, N0)")
        c0, ldc0 = C0.data_ptr(), _ld(C0, "C0")
    if beta1 != 0.0:
        if C1 is None or C1.dtype != torch.float32 or tuple(C1.shape) != (M, N1):
            raise ValueError("beta1 != 0 needs an fp32 C1 of shape (M, N1)")
        c1, ldc1 = C1.data_ptr(), _ld(C1, "C1")
    st = library().mp_gemm_b2b(h.ptr, M, N0, N1, K0, A0.data_ptr(), _ld(A0, "A0"), W0.data_ptr(), _ld(W0, "W0"),
                               c0, ldc0, W1.data_ptr(), _ld(W1, "W1"), c1, ldc1, D1.data_ptr(), _ld(D1, "D1"),
                               float(alpha0), float(beta0), float(alpha1), float(beta1), int(act0),
                               _stream_ptr(stream))
    _check(st, "mp_gemm_b2b")


MP_B2B_AUTO, MP_B2B_FUSED, MP_B2B_TWO_LAUNCH = 0, 1, 2


def mp_set_b2b_mode(h: Handle, mode: int) -> None:
    """MP_B2B_AUTO (default), MP_B2B_FUSED or MP_B2B_TWO_LAUNCH for mp_gemm_b2b."""
    _check(library().mp_set_b2b_mode(h.ptr, int(mode)), "mp_set_b2b_mode")


def mp_plan_b2b(h: Handle, M: int, N0: int, N1: int, K0: int) -> MpB2BPlan:
    """How mp_gemm_b2b splits an (M, N0, N1, K0) problem (host only)."""
    out = MpB2BPlan()
    _check(library().mp_plan_b2b(h.ptr, M, N0, N1, K0, ctypes.byref(out)), "mp_plan_b2b")
    return out


def _problems(items):
    """(A, B, C, D, alpha, beta) tuples of torch tensors -> MpGemmProblem array."""
    arr = (MpGemmProblem * max(1, len(items)))()
    for i, (A, B, C, D, alpha, beta) in enumerate(items):
        M, N, K, c_ptr, ldc = _gemm_args(A, B, C, D, beta)
        arr[i] = MpGemmProblem(M, N, K, A.data_ptr(), _ld(A, "A"), B.data_ptr(), _ld(B, "B"), c_ptr, ldc,
                               D.data_ptr(), _ld(D, "D"), float(alpha), float(beta))
    return arr


def mp_gemm_grouped(h: Handle, items, stream=None) -> None:
    """Every D_i = alpha_i*A_i@B_i + beta_i*C_i of a group of problems of any
    shapes, in as few launches as possible.  `items`: (A, B, C, D, alpha, beta)."""
    arr = _problems(items)
    _check(library().mp_gemm_grouped(h.ptr, len(items), arr, _stream_ptr(stream)), "mp_gemm_grouped")


def mp_plan_grouped(h: Handle, shapes) -> MpGroupedPlan:
    """The plan of a group given as (M, N, K) shapes (host only; no operands
    are read: the pointers are placeholders laid out without overlap)."""
    arr = (MpGemmProblem * max(1, len(shapes)))()
    base = 1 << 20
    for i, (M, N, K) in enumerate(shapes):
        a = base
        b = a + 2 * M * K + 256
        d = b + 2 * K * N + 256
        base = d + 4 * M * N + 256
        arr[i] = MpGemmProblem(M, N, K, a, max(K, 1), b, max(N, 1), None, 0, d, max(N, 1), 1.0, 0.0)
    out = MpGroupedPlan()
    _check(library().mp_plan_grouped(h.ptr, len(shapes), arr, ctypes.byref(out)), "mp_plan_grouped")
    return out


def _pixel_pitch(t, name, K):
    """Elements from one output pixel to the next of a [N, P, Q, K] tensor
    whose pixels are evenly spaced (NHWC, channels possibly padded)."""
    if t.dim() != 4 or (t.size(3) > 1 and t.stride(3) != 1):
        raise ValueError(f"{name} must be [N, P, Q, K] with unit channel stride")
    N, P, Q, _ = t.shape
    ld = t.stride(2) if Q > 1 else (t.stride(1) if P > 1 else (t.stride(0) if N > 1 else K))
    if (Q > 1 and t.stride(1) != Q * ld and P > 1) or (P * Q > 1 and N > 1 and t.stride(0) != P * Q * ld):
        raise ValueError(f"{name} pixels must be evenly spaced")
    return max(ld, K)


def mp_conv2d(h: Handle, X, F, Cin, D, alpha: float = 1.0, beta: float = 0.0, pad_h: int = 1, pad_w: int = 1,
              stream=None) -> None:
    """D = alpha * conv2d(X, F) + beta * Cin, stride 1, zero padding, NHWC, as an
    implicit GEMM.  X [N,H,W,C] and F [R,S,C,K] contiguous bfloat16; Cin and D
    [N,P,Q,K] float32."""
    import torch
    if X.dtype != torch.bfloat16 or F.dtype != torch.bfloat16 or X.dim() != 4 or F.dim() != 4:
        raise TypeError("X [N,H,W,C] and F [R,S,C,K] must be bfloat16")
    if not (X.is_contiguous() and F.is_contiguous()):
        raise ValueError("X and F must be contiguous")
    if D.dtype != torch.float32:
        raise TypeError("D must be float32")
    N, H, W, C = X.shape
    R, S, C2, K = F.shape
    P, Q = H + 2 * pad_h - R + 1, W + 2 * pad_w - S + 1
    if C2 != C or tuple(D.shape) != (N, P, Q, K):
        raise ValueError("shape mismatch")
    c_ptr, ldc = None, 0
    if beta != 0.0:
        if Cin is None or Cin.dtype != torch.float32 or tuple(Cin.shape) != (N, P, Q, K):
            raise ValueError("beta != 0 needs an fp32 Cin of D's shape")
        c_ptr, ldc = Cin.data_ptr(), _pixel_pitch(Cin, "Cin", K)
    st = library().mp_conv2d(h.ptr, N, H, W, C, K, R, S, pad_h, pad_w, X.data_ptr(), F.data_ptr(), c_ptr, ldc,
                             D.data_ptr(), _pixel_pitch(D, "D", K), float(alpha), float(beta), _stream_ptr(stream))
    _check(st, "mp_conv2d")


def mp_plan_conv(h: Handle, N: int, H: int, W: int, C: int, K: int, R: int = 3, S: int = 3, pad_h: int = 1,
                 pad_w: int = 1) -> MpConvPlan:
    """How mp_conv2d tiles a problem (host only)."""
    out = MpConvPlan()
    _check(library().mp_plan_conv(h.ptr, N, H, W, C, K, R, S, pad_h, pad_w, ctypes.byref(out)), "mp_plan_conv")
    return out


def mp_enumerate_plans(h: Handle, M: int, N: int, K: int, capacity=None, batch: int = 1):
    """The candidate strategies of one shape, cheapest first under the handle's
    cost model (all of them when capacity is None)."""
    n = ctypes.c_int32(0)
    lib = library()
    if capacity is None:
        _check(lib.mp_enumerate_plans(h.ptr, batch, M, N, K, None, 0, ctypes.byref(n)), "mp_enumerate_plans")
        capacity = n.value
    arr = (MpPlanInfo * max(1, capacity))()
    _check(lib.mp_enumerate_plans(h.ptr, batch, M, N, K, arr, capacity, ctypes.byref(n)), "mp_enumerate_plans")
    return [arr[i] for i in range(min(capacity, n.value))]


def mp_set_plan_mode(h: Handle, mode: int) -> None:
    """MP_PLAN_MIKPOLY (default), MP_PLAN_WAVE or MP_PLAN_PIPE cost model."""
    _check(library().mp_set_plan_mode(h.ptr, int(mode)), "mp_set_plan_mode")


def mp_gemm_batched(h: Handle, A, B, C, D, alpha: float = 1.0, beta: float = 0.0, stream=None) -> None:
    """Batched form on 3-D tensors [batch, rows, cols]; a batch stride of 0 shares an operand."""
    import torch
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16 or D.dtype != torch.float32:
        raise TypeError("A and B must be bfloat16, D float32")
    if A.dim() != 3 or B.dim() != 3 or D.dim() != 3:
        raise ValueError("batched operands are 3-D")
    batch = D.shape[0]
    M, K = A.shape[-2], A.shape[-1]
    N = B.shape[-1]
    sa = A.stride(0) if A.shape[0] > 1 else 0
    sb = B.stride(0) if B.shape[0] > 1 else 0
    c_ptr, ldc, sc = None, 0, 0
    if beta != 0.0:
        c_ptr, ldc = C.data_ptr(), _ld(C, "C")
        sc = C.stride(0) if C.shape[0] > 1 else 0
    st = library().mp_gemm_batched(h.ptr, batch, M, N, K, A.data_ptr(), _ld(A, "A"), sa,
                                   B.data_ptr(), _ld(B, "B"), sb, c_ptr, ldc, sc,
                                   D.data_ptr(), _ld(D, "D"), D.stride(0),
                                   float(alpha), float(beta), _stream_ptr(stream))
    _check(st, "mp_gemm_batched")


def mp_gemm_noalloc(A, B, C, D, alpha: float = 1.0, beta: float = 0.0, stream=None) -> None:
    """mp_gemm without a handle: for callers that cannot allocate device memory.

    The library keeps this call's scratch in a fixed array it owns (about
    48 MiB per GPU, held until exit); see mp_gemm_noalloc in include/mp.h.
    Calls that overlap on the GPU share that array and race.
    """
    import torch
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16 or D.dtype != torch.float32:
        raise TypeError("A and B must be bfloat16, D float32")
    M, K = A.shape[-2], A.shape[-1]
    N = B.shape[-1]
    if B.shape[-2] != K or D.shape[-2:] != (M, N):
        raise ValueError("shape mismatch")
    c_ptr, ldc = None, 0
    if beta != 0.0:
        if C is None or C.dtype != torch.float32 or C.shape[-2:] != (M, N):
            raise ValueError("beta != 0 needs an fp32 C of D's shape")
        c_ptr, ldc = C.data_ptr(), _ld(C, "C")
    st = library().mp_gemm_noalloc(M, N, K, A.data_ptr(), _ld(A, "A"), B.data_ptr(), _ld(B, "B"),
                                   c_ptr, ldc, D.data_ptr(), _ld(D, "D"), float(alpha), float(beta),
                                   _stream_ptr(stream))
    _check(st, "mp_gemm_noalloc")


def mp_check(h: Handle, stream=None) -> int:
    """Synchronize and return the device status (MP_OK or MP_ERR_DEVICE_TIMEOUT)."""
    return int(library().mp_check(h.ptr, _stream_ptr(stream)))


def mp_force_plan(h: Handle, kernel: int = -1, splits: int = 0) -> None:
    _check(library().mp_force_plan(h.ptr, kernel, splits), "mp_force_plan")


def mp_get_hw(h: Handle):
    hw = MpHw()
    ks = (MpKernelDesc * MP_MAX_KERNELS)()
    n = _i32()
    _check(library().mp_get_hw(h.ptr, ctypes.byref(hw), ks, ctypes.byref(n)), "mp_get_hw")
    return hw, [ks[i] for i in range(n.value)]


def mp_set_kernel_model(h: Handle, k: int, fixed_us: float, per_step_us: float, tail_us: float = 0.0) -> None:
    _check(library().mp_set_kernel_model(h.ptr, k, fixed_us, per_step_us, tail_us), "mp_set_kernel_model")


def mp_set_split_model(h: Handle, on_chip: int, sync_us: float, bytes_factor: float, S: int = 0) -> None:
    """on_chip 0: the reduction through L2 (S 0); 1: on chip in clusters of S
    (2..8), or every cluster size when S is 0."""
    _check(library().mp_set_split_model(h.ptr, int(on_chip), int(S), sync_us, bytes_factor), "mp_set_split_model")


def mp_load_calibration(h: Handle, path: str) -> None:
    _check(library().mp_load_calibration(h.ptr, os.fsencode(path)), "mp_load_calibration")


def mp_get_split_model(h: Handle, on_chip: int, S: int = 0):
    """(sync_us, bytes_factor) of the split-K reduction: on_chip 0 (S 0)
    through L2, on_chip 1 on chip in clusters of S (2..8)."""
    s, f = ctypes.c_double(), ctypes.c_double()
    _check(library().mp_get_split_model(h.ptr, int(on_chip), int(S), ctypes.byref(s), ctypes.byref(f)),
           "mp_get_split_model")
    return s.value, f.value


def mp_inject_wait_timeout(h: Handle, enable=True, limit_ns: int = 0) -> None:
    """enable: True or 1 withholds a pipeline stage of the next launch; 2 makes
    the GEMM kernel's ring-staged split-K sums wait for bytes that never come;
    False or 0 clears it."""
    _check(library().mp_inject_wait_timeout(h.ptr, int(enable), int(limit_ns)),
           "mp_inject_wait_timeout")


def mp_check_noalloc(stream=None) -> int:
    """mp_check for mp_gemm_noalloc on the current device (no handle)."""
    return int(library().mp_check_noalloc(_stream_ptr(stream)))


def mp_noalloc_inject_wait_timeout(enable=True, limit_ns: int = 0) -> None:
    _check(library().mp_noalloc_inject_wait_timeout(int(enable), int(limit_ns)),
           "mp_noalloc_inject_wait_timeout")

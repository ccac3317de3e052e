"""Thin ctypes binding of libgemm15.so -- argument marshalling only.

Every function here has the name of the C entry point it calls
(include/gemm15.h) and does nothing but convert arguments: torch tensors
become device pointers, torch streams become cudaStream_t.  All arithmetic
runs in the library's CUDA kernels; if the library cannot be loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

# enums mirrored from include/gemm15.h
F16, BF16, F32, E4M3, E5M2, E2M1 = 0, 1, 2, 3, 4, 5
SCALE_MX, SCALE_NV = 1, 2
ROW_MAJOR, COL_MAJOR = 0, 1
EPI_LINEAR, EPI_RELU, EPI_SIGMOID, EPI_TANH = 0, 1, 2, 3
EPILOGUES = {"linear": EPI_LINEAR, "relu": EPI_RELU, "sigmoid": EPI_SIGMOID, "tanh": EPI_TANH}
AUX_OPS = {None: 0, "add": 1, "sub": 2, "mul": 3, "div": 4}
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIGNMENT, ERR_CUDA, ERR_TIMEOUT, ERR_OOM, \
    ERR_DEVICE_FAULT, ERR_NO_DEVICE, ERR_BAD_PLAN = range(10)
OPT_SCHEDULE, OPT_SPLITS, OPT_CTA_GROUP, OPT_TILE_N, OPT_RASTER, OPT_GRID, \
    OPT_TIMEOUT_US, OPT_FAULT_SKIP_FLAG, OPT_SK_DP_WAVES, OPT_TRACE_ITEMS, OPT_SWAP_AB, \
    OPT_SPLITK_INLINE, OPT_L2_HINTS = range(13)
SCHED_AUTO, SCHED_DP, SCHED_SK, SCHED_SPLIT = range(4)

DTYPES = {"f16": F16, "bf16": BF16, "f32": F32, "e4m3": E4M3, "e5m2": E5M2, "e2m1": E2M1}

EXPORTED = (
    "gemm_plan_create", "gemm_plan_destroy", "gemm_run", "gemm_run_ex", "gemm_run_host",
    "grouped_gemm_run", "gemm_plan_query_error", "gemm15_status_string",
    "gemm_plan_set_option", "gemm_plan_last_config", "gemm_run_splitk_noalloc",
    "gemm_plan_trace", "gemm_run_batched", "gemm_run_args", "gemm_plan_autotune",
    "gemm_plan_forget_tuning", "gemm_run_block_scaled",
)


class PlanDesc(ctypes.Structure):
    _fields_ = [("a", ctypes.c_int), ("b", ctypes.c_int), ("c", ctypes.c_int),
                ("d", ctypes.c_int), ("acc", ctypes.c_int), ("layout_a", ctypes.c_int),
                ("layout_b", ctypes.c_int), ("layout_cd", ctypes.c_int),
                ("epilogue", ctypes.c_int)]


class Args(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("lda", ctypes.c_int64), ("B", ctypes.c_void_p),
                ("ldb", ctypes.c_int64), ("C", ctypes.c_void_p), ("ldc", ctypes.c_int64),
                ("D", ctypes.c_void_p), ("ldd", ctypes.c_int64), ("M", ctypes.c_int64),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("alpha", ctypes.c_float),
                ("beta", ctypes.c_float), ("scale_a", ctypes.c_void_p),
                ("scale_b", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("aux", ctypes.c_void_p), ("ldaux", ctypes.c_int64), ("aux_op", ctypes.c_int32),
                ("pre", ctypes.c_void_p), ("ldpre", ctypes.c_int64)]


class ScaledArgs(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("lda", ctypes.c_int64), ("B", ctypes.c_void_p),
                ("ldb", ctypes.c_int64), ("SFA", ctypes.c_void_p), ("SFB", ctypes.c_void_p),
                ("scale_kind", ctypes.c_int32), ("C", ctypes.c_void_p), ("ldc", ctypes.c_int64),
                ("D", ctypes.c_void_p), ("ldd", ctypes.c_int64), ("M", ctypes.c_int64),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("alpha", ctypes.c_float),
                ("beta", ctypes.c_float), ("bias", ctypes.c_void_p)]


class Problem(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("C", ctypes.c_void_p),
                ("D", ctypes.c_void_p), ("lda", ctypes.c_int64), ("ldb", ctypes.c_int64),
                ("ldc", ctypes.c_int64), ("ldd", ctypes.c_int64),
                ("scale_a", ctypes.c_void_p), ("scale_b", ctypes.c_void_p)]


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "cta_group", "tile_m", "tile_n", "tile_k", "stages", "schedule", "grid", "tiles",
        "splits", "raster", "launches", "swap_ab")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class TuneResult(ctypes.Structure):
    _fields_ = [("config", Config), ("sk_dp_waves", ctypes.c_int32), ("us", ctypes.c_float),
                ("status", ctypes.c_int)]

    def as_dict(self):
        return {"config": self.config.as_dict(), "sk_dp_waves": self.sk_dp_waves,
                "us": self.us, "status": self.status}


class Gemm15Error(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what or "gemm15", status_string(status), status))


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Loads libgemm15.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build() if build_if_missing else _build.LIB
        if not os.path.exists(path):
            raise RuntimeError("libgemm15.so is not built (%s); run dense_gemm_15_gb300.build.build()" % path)
        lib = ctypes.CDLL(path)
        i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
        st = ctypes.c_int
        lib.gemm_plan_create.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(PlanDesc)]
        lib.gemm_plan_destroy.argtypes = [vp]
        lib.gemm_run.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, f32, f32, vp]
        lib.gemm_run_ex.argtypes = [vp, vp, i64, vp, i64, vp, i64, vp, i64, i64, i64, i64,
                                    f32, f32, vp, vp, vp]
        lib.gemm_run_host.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, f32, f32, f32, f32, vp]
        lib.grouped_gemm_run.argtypes = [vp, ctypes.POINTER(Problem), i32, f32, f32, vp]
        lib.gemm_run_args.argtypes = [vp, ctypes.POINTER(Args), vp]
        lib.gemm_plan_autotune.argtypes = [vp, ctypes.POINTER(Args), i32,
                                           ctypes.POINTER(TuneResult), i32,
                                           ctypes.POINTER(i32), vp]
        lib.gemm_plan_forget_tuning.argtypes = [vp]
        lib.gemm_run_block_scaled.argtypes = [vp, ctypes.POINTER(ScaledArgs), vp]
        lib.gemm_run_batched.argtypes = [vp, vp, i64, i64, vp, i64, i64, vp, i64, i64, vp, i64,
                                         i64, i64, i64, i64, i32, f32, f32, vp]
        lib.gemm_plan_query_error.argtypes = [vp]
        lib.gemm15_status_string.argtypes = [st]
        lib.gemm15_status_string.restype = ctypes.c_char_p
        lib.gemm_plan_set_option.argtypes = [vp, st, i64]
        lib.gemm_plan_last_config.argtypes = [vp, ctypes.POINTER(Config)]
        lib.gemm_plan_trace.argtypes = [vp, vp, i64, ctypes.POINTER(i32), ctypes.POINTER(i32)]
        lib.gemm_run_splitk_noalloc.argtypes = [ctypes.POINTER(PlanDesc), vp, i64, vp, i64, vp,
                                                i64, vp, i64, i64, i64, i64, f32, f32, vp, vp,
                                                i32, vp, vp]
        for name in EXPORTED:
            if name != "gemm15_status_string":
                getattr(lib, name).restype = st
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().gemm15_status_string(int(status)).decode()


def _check(status, what):
    if status != OK:
        raise Gemm15Error(status, what)
    return status


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------------ raw C calls

def gemm_plan_create(a="f16", b=None, c=None, d=None, acc="f32", layout_a=ROW_MAJOR,
                     layout_b=ROW_MAJOR, layout_cd=ROW_MAJOR, relu=False, epilogue=None):
    """epilogue: "linear", "relu", "sigmoid", "tanh" (or its code); default from relu."""
    lib = load()
    b = b or a
    c = c or ("bf16" if a == "e4m3" else a)
    d = d or c
    if epilogue is None:
        epi = EPI_RELU if relu else EPI_LINEAR
    else:
        epi = EPILOGUES[epilogue] if isinstance(epilogue, str) else int(epilogue)
    desc = PlanDesc(DTYPES[a], DTYPES[b], DTYPES[c], DTYPES[d], DTYPES[acc], layout_a,
                    layout_b, layout_cd, epi)
    h = ctypes.c_void_p()
    _check(lib.gemm_plan_create(ctypes.byref(h), ctypes.byref(desc)), "gemm_plan_create")
    return h.value


def gemm_plan_destroy(plan):
    return _check(load().gemm_plan_destroy(plan), "gemm_plan_destroy")


def gemm_run(plan, A, B, C, D, M, N, K, alpha=1.0, beta=0.0, stream=None):
    return load().gemm_run(plan, _ptr(A), _ptr(B), _ptr(C), _ptr(D), M, N, K, alpha, beta,
                           _stream(stream))


def gemm_run_ex(plan, A, lda, B, ldb, C, ldc, D, ldd, M, N, K, alpha=1.0, beta=0.0,
                scale_a=None, scale_b=None, stream=None):
    return load().gemm_run_ex(plan, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, _ptr(D), ldd,
                              M, N, K, alpha, beta, _ptr(scale_a), _ptr(scale_b),
                              _stream(stream))


def gemm_run_host(plan, hA, hB, hC, hD, M, N, K, alpha=1.0, beta=0.0, scale_a=1.0,
                  scale_b=1.0, stream=None):
    return load().gemm_run_host(plan, _ptr(hA), _ptr(hB), _ptr(hC), _ptr(hD), M, N, K, alpha,
                                beta, scale_a, scale_b, _stream(stream))


def grouped_gemm_run(plan, problems, alpha=1.0, beta=0.0, stream=None):
    """problems: sequence of (M, N, K, A, B, C, D) or dicts with optional ld*
    and, for e4m3 plans, scale_a / scale_b (device float tensors)."""
    arr = (Problem * max(len(problems), 1))()
    for i, pr in enumerate(problems):
        if isinstance(pr, dict):
            q = pr
        else:
            q = dict(zip(("M", "N", "K", "A", "B", "C", "D"), pr))
        arr[i] = Problem(q["M"], q["N"], q["K"], _ptr(q["A"]), _ptr(q["B"]), _ptr(q.get("C")),
                         _ptr(q["D"]), q.get("lda", 0), q.get("ldb", 0), q.get("ldc", 0),
                         q.get("ldd", 0), _ptr(q.get("scale_a")), _ptr(q.get("scale_b")))
    return load().grouped_gemm_run(plan, arr, len(problems), alpha, beta, _stream(stream))


def gemm_run_args(plan, A, B, C, D, M, N, K, alpha=1.0, beta=0.0, lda=0, ldb=0, ldc=0, ldd=0,
                  scale_a=None, scale_b=None, bias=None, aux=None, ldaux=0, aux_op=None,
                  pre=None, ldpre=0, stream=None):
    """aux_op: None, "add", "sub", "mul", "div" (or its code); pre: optional
    output of the pre-activation value."""
    op = AUX_OPS[aux_op] if aux_op is None or isinstance(aux_op, str) else int(aux_op)
    args = Args(_ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, _ptr(D), ldd, M, N, K, alpha, beta,
                _ptr(scale_a), _ptr(scale_b), _ptr(bias), _ptr(aux), ldaux, op, _ptr(pre), ldpre)
    return load().gemm_run_args(plan, ctypes.byref(args), _stream(stream))


def gemm_plan_autotune(plan, A, B, C, D, M, N, K, alpha=1.0, beta=0.0, lda=0, ldb=0, ldc=0,
                       ldd=0, scale_a=None, scale_b=None, bias=None, iterations=10,
                       stream=None):
    """Returns (status, [result dicts, fastest first])."""
    args = Args(_ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, _ptr(D), ldd, M, N, K, alpha, beta,
                _ptr(scale_a), _ptr(scale_b), _ptr(bias), None, 0, 0, None, 0)
    cap = 64
    out = (TuneResult * cap)()
    n = ctypes.c_int32()
    st = load().gemm_plan_autotune(plan, ctypes.byref(args), int(iterations), out, cap,
                                   ctypes.byref(n), _stream(stream))
    return st, [out[i].as_dict() for i in range(min(n.value, cap))]


def gemm_run_block_scaled(plan, A, B, SFA, SFB, D, M, N, K, scale_kind=SCALE_MX, C=None,
                          alpha=1.0, beta=0.0, lda=0, ldb=0, ldc=0, ldd=0, bias=None,
                          stream=None):
    """Block-scaled GEMM (A row-major, B column-major, scale factors in the
    128 x 4 blocked layout; see include/gemm15.h)."""
    args = ScaledArgs(_ptr(A), lda, _ptr(B), ldb, _ptr(SFA), _ptr(SFB), int(scale_kind), _ptr(C),
                      ldc, _ptr(D), ldd, M, N, K, alpha, beta, _ptr(bias))
    return load().gemm_run_block_scaled(plan, ctypes.byref(args), _stream(stream))


def gemm_plan_forget_tuning(plan):
    return load().gemm_plan_forget_tuning(plan)


def gemm_run_batched(plan, A, lda, stride_a, B, ldb, stride_b, C, ldc, stride_c, D, ldd,
                     stride_d, M, N, K, batch, alpha=1.0, beta=0.0, stream=None):
    return load().gemm_run_batched(plan, _ptr(A), lda, stride_a, _ptr(B), ldb, stride_b,
                                   _ptr(C), ldc, stride_c, _ptr(D), ldd, stride_d, M, N, K,
                                   batch, alpha, beta, _stream(stream))


def gemm_plan_query_error(plan):
    return load().gemm_plan_query_error(plan)


def gemm_plan_set_option(plan, option, value):
    return _check(load().gemm_plan_set_option(plan, option, int(value)), "gemm_plan_set_option")


def gemm_plan_last_config(plan):
    cfg = Config()
    _check(load().gemm_plan_last_config(plan, ctypes.byref(cfg)), "gemm_plan_last_config")
    return cfg.as_dict()


def gemm_plan_trace(plan):
    """Timeline of the plan's last traced launch: uint64 array [ctas, 1 + items, 8]."""
    import numpy as np
    lib = load()
    ctas, items = ctypes.c_int32(), ctypes.c_int32()
    lib.gemm_plan_trace(plan, None, 0, ctypes.byref(ctas), ctypes.byref(items))
    out = np.zeros((max(ctas.value, 0), max(items.value, 0) + 1, 8), dtype=np.uint64)
    _check(lib.gemm_plan_trace(plan, out.ctypes.data, out.nbytes, ctypes.byref(ctas),
                               ctypes.byref(items)), "gemm_plan_trace")
    return out


def gemm_run_splitk_noalloc(a, layout_a, layout_b, layout_cd, relu, A, lda, B, ldb, C, ldc, D,
                            ldd, M, N, K, alpha=1.0, beta=0.0, scale_a=None, scale_b=None,
                            splits=1, status=None, stream=None):
    """Split-K GEMM that allocates no device memory (see include/gemm15.h)."""
    c = "bf16" if a == "e4m3" else a
    desc = PlanDesc(DTYPES[a], DTYPES[a], DTYPES[c], DTYPES[c], F32, layout_a, layout_b,
                    layout_cd, EPI_RELU if relu else EPI_LINEAR)
    return load().gemm_run_splitk_noalloc(ctypes.byref(desc), _ptr(A), lda, _ptr(B), ldb,
                                          _ptr(C), ldc, _ptr(D), ldd, M, N, K, alpha, beta,
                                          _ptr(scale_a), _ptr(scale_b), int(splits),
                                          _ptr(status), _stream(stream))


# ------------------------------------------------------------------ convenience

class Plan:
    """A plan bound to element types and layouts; run() takes torch CUDA tensors.

    Mirrors the plan object of the CUTLASS Python interface: types and layouts
    are fixed at construction, any shape may be run later."""

    def __init__(self, dtype="f16", out_dtype=None, relu=False, layout_a=ROW_MAJOR,
                 layout_b=ROW_MAJOR, layout_cd=ROW_MAJOR, epilogue=None):
        self.dtype = dtype
        self.out_dtype = out_dtype or ("bf16" if dtype == "e4m3" else dtype)
        self.layouts = (layout_a, layout_b, layout_cd)
        self.handle = gemm_plan_create(dtype, dtype, self.out_dtype, self.out_dtype, "f32",
                                       layout_a, layout_b, layout_cd, relu, epilogue)

    def close(self):
        if self.handle:
            gemm_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set(self, option, value):
        gemm_plan_set_option(self.handle, option, value)
        return self

    def run(self, A, B, C, D, M=None, N=None, K=None, alpha=1.0, beta=0.0, scale_a=None,
            scale_b=None, stream=None, lda=None, ldb=None, ldc=None, ldd=None, bias=None,
            aux=None, aux_op=None, ldaux=0):
        la, lb, lcd = self.layouts
        if M is None:
            M = A.shape[0] if la == ROW_MAJOR else A.shape[1]
            K = A.shape[1] if la == ROW_MAJOR else A.shape[0]
            N = B.shape[1] if lb == ROW_MAJOR else B.shape[0]
        lda = lda or (K if la == ROW_MAJOR else M)
        ldb = ldb or (N if lb == ROW_MAJOR else K)
        ldd = ldd or (N if lcd == ROW_MAJOR else M)
        ldc = ldc or ldd
        if bias is not None or aux_op is not None:
            st = gemm_run_args(self.handle, A, B, C, D, M, N, K, alpha, beta, lda, ldb, ldc, ldd,
                               scale_a, scale_b, bias, aux, ldaux, aux_op, stream)
        else:
            st = gemm_run_ex(self.handle, A, lda, B, ldb, C, ldc, D, ldd, M, N, K, alpha, beta,
                             scale_a, scale_b, stream)
        _check(st, "gemm_run")
        return D

    def grouped(self, problems, alpha=1.0, beta=0.0, stream=None):
        _check(grouped_gemm_run(self.handle, problems, alpha, beta, stream), "grouped_gemm_run")

    def batched(self, A, B, C, D, M, N, K, batch, stride_a, stride_b, stride_c, stride_d,
                alpha=1.0, beta=0.0, lda=0, ldb=0, ldc=0, ldd=0, stream=None):
        """Uniform-stride batch of one shape (strides in elements; 0 shares an operand)."""
        _check(gemm_run_batched(self.handle, A, lda, stride_a, B, ldb, stride_b, C, ldc,
                                stride_c, D, ldd, stride_d, M, N, K, batch, alpha, beta,
                                stream), "gemm_run_batched")
        return D

    def autotune(self, A, B, C, D, M, N, K, alpha=1.0, beta=0.0, bias=None, scale_a=None,
                 scale_b=None, iterations=10, stream=None, **ld):
        """Times every candidate kernel configuration for this shape and keeps the
        fastest for later runs of the same (M, N, K); returns the results."""
        st, res = gemm_plan_autotune(self.handle, A, B, C, D, M, N, K, alpha, beta,
                                     ld.get("lda", 0), ld.get("ldb", 0), ld.get("ldc", 0),
                                     ld.get("ldd", 0), scale_a, scale_b, bias, iterations,
                                     stream)
        _check(st, "gemm_plan_autotune")
        return res

    def query_error(self):
        return gemm_plan_query_error(self.handle)

    def last_config(self):
        return gemm_plan_last_config(self.handle)

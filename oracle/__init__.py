"""CPU oracle for the dense GEMM hot path -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU product path never does, and
this package imports nothing from it: the two share no code.

The arithmetic lives in ``gemm_oracle.c`` (a plain fp64 triple loop, see its
header for the definition it follows and the passages it cites); this module
only compiles it with gcc and marshals numpy arrays into it.

Operands are passed as the raw stored bits (uint16 for fp16 / bf16, uint8 for
e4m3, float32 / float64 as themselves), in a 2-D numpy array that is the
matrix's storage: for a row-major M x K operand an (M, K) array, for a
column-major one the (K, M) array holding its transpose row by row.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F16, BF16, F32, E4M3, F64, E5M2, E2M1, UE8M0 = 0, 1, 2, 3, 4, 5, 6, 7
ACTS = {"linear": 0, "relu": 1, "sigmoid": 2, "tanh": 3}
AUX_OPS = {None: 0, "add": 1, "sub": 2, "mul": 3, "div": 4}
_NAMES = {"f16": F16, "bf16": BF16, "f32": F32, "e4m3": E4M3, "f64": F64, "e5m2": E5M2,
          "e2m1": E2M1, "ue8m0": UE8M0}
_ITEMSIZE = {F16: 2, BF16: 2, F32: 4, E4M3: 1, F64: 8, E5M2: 1, E2M1: 1, UE8M0: 1}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libgemm_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math: the sum order is the
    definition's).  Returns the library path."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                    "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"],
                   check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.oracle_gemm.restype = i32
            lib.oracle_gemm.argtypes = [vp, i32, i64, i32, vp, i32, i64, i32, vp, i32, i64,
                                        vp, i64, i64, i64, i64, dbl, dbl, dbl, dbl,
                                        i32, vp, i32, vp, i32, i64, i32, vp, vp, i32, i64,
                                        i32, i64, i64, i32]
            lib.oracle_round_f16_array.argtypes = [vp, vp, i64]
            lib.oracle_round_bf16_array.argtypes = [vp, vp, i64]
            lib.oracle_decode_array.argtypes = [vp, i32, vp, i64]
            _lib = lib
    return _lib


def dtype_code(dt) -> int:
    return _NAMES[dt] if isinstance(dt, str) else int(dt)


def _leading(arr: np.ndarray, code: int) -> int:
    if arr.ndim == 2 and arr.size == 0:
        return max(1, arr.shape[1])  # an empty operand (K == 0) is never read
    if arr.ndim != 2 or arr.strides[1] != _ITEMSIZE[code]:
        raise ValueError("operand storage must be 2-D with unit inner stride")
    if arr.strides[0] % _ITEMSIZE[code]:
        raise ValueError("row stride is not a whole number of elements")
    return arr.strides[0] // _ITEMSIZE[code]


def default_threads() -> int:
    return os.cpu_count() or 1


def gemm(a, a_dtype, b, b_dtype, c=None, c_dtype="f16", *, alpha=1.0, beta=0.0,
         relu=False, scale_a=1.0, scale_b=1.0, a_col_major=False, b_col_major=False,
         rows=None, threads=None, absolute=False, act=None, bias=None,
         bias_dtype=None, aux=None, aux_dtype=None, aux_op=None, scales=None) -> np.ndarray:
    """D = act(alpha * s_a * s_b * (A @ B) + beta * C + bias) in float64, for
    rows ``rows = (begin, end)`` of D (all rows by default).

    ``act`` is "linear", "relu", "sigmoid" or "tanh" (default: "relu" if
    ``relu`` else "linear"); ``bias`` is the stored bits of an N-vector of type
    ``bias_dtype`` (default ``c_dtype``), added to every row; ``aux`` (M x N
    row-major storage of type ``aux_dtype``, default ``c_dtype``) enters the
    activated value by ``aux_op`` in "add", "sub", "mul", "div".  ``scales`` =
    (SA, SB, scale_dtype, block) makes A and B block-scaled: SA is M x
    ceil(K/block), SB ceil(K/block) x N, both row-major stored bits.

    ``absolute=True`` returns sum_k |A[i,k]| |B[k,j]| instead (the matrix the
    error bound of the checker is built from); alpha/beta/C are then unused.
    """
    lib = _load()
    ac, bc = dtype_code(a_dtype), dtype_code(b_dtype)
    cc = dtype_code(c_dtype)
    a = np.asarray(a)
    b = np.asarray(b)
    if a_col_major:
        K, M = a.shape
    else:
        M, K = a.shape
    if b_col_major:
        N, Kb = b.shape
    else:
        Kb, N = b.shape
    if Kb != K:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, Kb))
    lda, ldb = _leading(a, ac), _leading(b, bc)
    if c is not None:
        c = np.asarray(c)
        if c.shape != (M, N):
            raise ValueError("C must be M x N row-major storage")
        ldc = _leading(c, cc)
        cptr = c.ctypes.data
    else:
        if beta != 0.0 and not absolute:
            raise ValueError("beta != 0 needs C")
        ldc, cptr = 0, None
    act_code = ACTS[act] if act is not None else (1 if relu else 0)
    bptr, bcode = None, 0
    if bias is not None:
        bias = np.ascontiguousarray(bias)
        if bias.shape != (N,):
            raise ValueError("bias must hold N elements")
        bcode = dtype_code(bias_dtype or c_dtype)
        bptr = bias.ctypes.data
    zptr, zcode, ldz, op = None, 0, 0, AUX_OPS[aux_op]
    if op:
        aux = np.asarray(aux)
        if aux.shape != (M, N):
            raise ValueError("aux must be M x N row-major storage")
        zcode = dtype_code(aux_dtype or c_dtype)
        ldz = _leading(aux, zcode)
        zptr = aux.ctypes.data
    sa_ptr = sb_ptr = None
    s_code, block = 0, 0
    if scales is not None:
        sa, sb, s_dt, block = scales
        kb = -(-K // block)
        sa, sb = np.ascontiguousarray(sa), np.ascontiguousarray(sb)
        if sa.shape != (M, kb) or sb.shape != (kb, N):
            raise ValueError("block scales must be M x ceil(K/block) and ceil(K/block) x N")
        s_code = dtype_code(s_dt)
        sa_ptr, sb_ptr = sa.ctypes.data, sb.ctypes.data
    r0, r1 = (0, M) if rows is None else rows
    out = np.empty((r1 - r0, N), dtype=np.float64)
    rc = lib.oracle_gemm(a.ctypes.data, ac, lda, int(a_col_major),
                         b.ctypes.data, bc, ldb, int(b_col_major),
                         cptr, cc, ldc, out.ctypes.data, N, M, N, K,
                         float(alpha), float(beta), float(scale_a), float(scale_b),
                         act_code, bptr, bcode, zptr, zcode, ldz, op, sa_ptr, sb_ptr, s_code,
                         int(block), int(bool(absolute)), r0, r1,
                         int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle_gemm failed with code %d" % rc)
    return out


def round_to(x: np.ndarray, dtype) -> np.ndarray:
    """Round float64 values to fp16 or bf16 bits (nearest, ties to even)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    code = dtype_code(dtype)
    if code == F16:
        lib.oracle_round_f16_array(x.ctypes.data, out.ctypes.data, x.size)
    elif code == BF16:
        lib.oracle_round_bf16_array(x.ctypes.data, out.ctypes.data, x.size)
    else:
        raise ValueError("round_to supports f16 and bf16")
    return out


def decode(bits: np.ndarray, dtype) -> np.ndarray:
    """Decode stored element bits to float64 exactly."""
    lib = _load()
    code = dtype_code(dtype)
    want = {F16: np.uint16, BF16: np.uint16, E4M3: np.uint8, F32: np.float32,
            F64: np.float64, E5M2: np.uint8, E2M1: np.uint8, UE8M0: np.uint8}[code]
    bits = np.ascontiguousarray(bits, dtype=want)
    out = np.empty(bits.shape, dtype=np.float64)
    lib.oracle_decode_array(bits.ctypes.data, code, out.ctypes.data, bits.size)
    return out

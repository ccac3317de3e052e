"""The C-ABI library loads and exports every entry point include/gemm15.h
declares; host-side argument checks behave as documented.  CPU only: no call
here reaches a kernel."""
import ctypes
import os
import re
import subprocess

import pytest

from dense_gemm_15_gb300 import binding as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "gemm15.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w[\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)))


def test_header_lists_expected_functions():
    names = header_functions()
    assert set(g.EXPORTED) == set(names), names


def test_library_exports_every_declared_symbol():
    lib = g.load()
    for name in header_functions():
        assert hasattr(lib, name), name


def test_status_strings():
    for s in range(10):
        txt = g.status_string(s)
        assert txt and txt != "unknown status"
    assert g.status_string(999) == "unknown status"


def test_null_plan_is_rejected_without_device():
    lib = g.load()
    assert lib.gemm_plan_destroy(None) == g.ERR_BAD_PLAN
    assert lib.gemm_run(None, None, None, None, None, 1, 1, 1, 1.0, 0.0, None) == g.ERR_BAD_PLAN
    assert lib.gemm_plan_query_error(None) == g.ERR_BAD_PLAN
    assert lib.gemm_plan_set_option(None, 0, 0) == g.ERR_BAD_PLAN
    assert lib.grouped_gemm_run(None, None, 0, 1.0, 0.0, None) == g.ERR_BAD_PLAN


def test_plan_create_argument_checks():
    lib = g.load()
    h = ctypes.c_void_p()
    assert lib.gemm_plan_create(None, None) == g.ERR_INVALID_ARG
    bad = g.PlanDesc(7, 0, 0, 0, 2, 0, 0, 0, 0)
    assert lib.gemm_plan_create(ctypes.byref(h), ctypes.byref(bad)) == g.ERR_INVALID_ARG
    mixed = g.PlanDesc(g.F16, g.BF16, g.F16, g.F16, g.F32, 0, 0, 0, 0)
    assert lib.gemm_plan_create(ctypes.byref(h), ctypes.byref(mixed)) == g.ERR_UNSUPPORTED
    acc16 = g.PlanDesc(g.F16, g.F16, g.F16, g.F16, g.F16, 0, 0, 0, 0)
    assert lib.gemm_plan_create(ctypes.byref(h), ctypes.byref(acc16)) == g.ERR_UNSUPPORTED
    f8_f16out = g.PlanDesc(g.E4M3, g.E4M3, g.F16, g.F16, g.F32, 0, 0, 0, 0)
    assert lib.gemm_plan_create(ctypes.byref(h), ctypes.byref(f8_f16out)) == g.ERR_UNSUPPORTED


def test_plan_create_without_gpu_reports_no_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    lib = g.load()
    h = ctypes.c_void_p()
    ok = g.PlanDesc(g.F16, g.F16, g.F16, g.F16, g.F32, 0, 0, 0, 0)
    assert lib.gemm_plan_create(ctypes.byref(h), ctypes.byref(ok)) == g.ERR_NO_DEVICE
    assert h.value is None


def test_binding_names_match_c_entry_points():
    for name in g.EXPORTED:
        if name == "gemm15_status_string":
            continue
        assert callable(getattr(g, name)), name


def test_ctypes_structs_match_the_header_layout(tmp_path):
    """Compile a probe against include/gemm15.h with the host C compiler and
    compare every struct's size and field offsets with the ctypes mirrors."""
    mirrors = {"gemm15_plan_desc_t": g.PlanDesc, "gemm15_problem_t": g.Problem,
               "gemm15_config_t": g.Config, "gemm15_args_t": g.Args,
               "gemm15_tune_result_t": g.TuneResult, "gemm15_scaled_args_t": g.ScaledArgs}
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "gemm15.h"', "int main(void) {"]
    for cname, cls in mirrors.items():
        lines.append('printf("%s size %%zu\\n", sizeof(%s));' % (cname, cname))
        for field, _ in cls._fields_:
            lines.append('printf("%s %s %%zu\\n", offsetof(%s, %s));' % (cname, field, cname, field))
    lines += ["return 0;", "}"]
    src = tmp_path / "probe.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {}
    for line in out:
        if line:
            parts = line.split()
            got[(parts[0], parts[1])] = int(parts[2])
    for cname, cls in mirrors.items():
        assert got[(cname, "size")] == ctypes.sizeof(cls), cname
        for field, _ in cls._fields_:
            assert got[(cname, field)] == getattr(cls, field).offset, (cname, field)


def test_noalloc_argument_checks_precede_any_device_call():
    """gemm_run_splitk_noalloc validates its descriptor, sizes and split count
    before it touches the device, so these answers need no GPU."""
    lib = g.load()

    def call(desc, M=64, N=64, K=64, splits=2, scale=None):
        d = ctypes.byref(desc) if desc is not None else None
        return lib.gemm_run_splitk_noalloc(d, None, K, None, N, None, N, None, N, M, N, K, 1.0,
                                           0.0, scale, None, splits, None, None)

    ok = g.PlanDesc(g.F16, g.F16, g.F16, g.F16, g.F32, 0, 0, 0, 0)
    assert call(None) == g.ERR_INVALID_ARG
    assert call(g.PlanDesc(g.F16, g.BF16, g.F16, g.F16, g.F32, 0, 0, 0, 0)) == g.ERR_UNSUPPORTED
    assert call(g.PlanDesc(g.F16, g.F16, g.F16, g.F16, g.F16, 0, 0, 0, 0)) == g.ERR_UNSUPPORTED
    assert call(g.PlanDesc(g.E4M3, g.E4M3, g.F16, g.F16, g.F32, 0, 0, 0, 0)) == g.ERR_UNSUPPORTED
    assert call(g.PlanDesc(g.F16, g.F16, g.F16, g.F16, g.F32, 2, 0, 0, 0)) == g.ERR_INVALID_ARG
    assert call(g.PlanDesc(g.F16, g.F16, g.F16, g.F16, g.F32, 0, 0, 0, 9)) == g.ERR_INVALID_ARG
    scale = ctypes.c_float(1.0)
    assert call(ok, scale=ctypes.addressof(scale)) == g.ERR_INVALID_ARG  # scales are fp8-only
    assert call(ok, splits=0) == g.ERR_INVALID_ARG
    assert call(ok, M=-1) == g.ERR_INVALID_ARG
    assert call(ok, K=1 << 31) == g.ERR_INVALID_ARG
    assert call(ok, M=0) == g.OK and call(ok, N=0) == g.OK  # nothing to do


def test_noalloc_pointer_and_layout_checks_precede_any_device_call():
    """Null D, a missing C with beta != 0, leading dimensions below the
    extent, misaligned pointers or leading dimensions and a problem beyond the
    scratch are answered before any device call (host addresses stand in for
    device ones: nothing is dereferenced)."""
    lib = g.load()
    ok = g.PlanDesc(g.F16, g.F16, g.F16, g.F16, g.F32, 0, 0, 0, 0)
    buf = ctypes.create_string_buffer(4096 + 64)
    base = (ctypes.addressof(buf) + 63) // 64 * 64

    def call(A=base, lda=64, B=base, ldb=64, C=None, ldc=64, D=base, ldd=64, M=64, N=64, K=64,
             beta=0.0, splits=2, desc=ok):
        return lib.gemm_run_splitk_noalloc(ctypes.byref(desc), A, lda, B, ldb, C, ldc, D, ldd,
                                           M, N, K, 1.0, beta, None, None, splits, None, None)

    assert call(D=None) == g.ERR_INVALID_ARG
    assert call(beta=1.0) == g.ERR_INVALID_ARG                 # C missing
    assert call(A=None) == g.ERR_INVALID_ARG
    assert call(ldd=32) == g.ERR_INVALID_ARG                   # below N
    assert call(lda=32) == g.ERR_INVALID_ARG                   # below K
    assert call(ldd=68) == g.ERR_ALIGNMENT                     # 136 bytes
    assert call(D=base + 2) == g.ERR_ALIGNMENT
    assert call(A=base + 8) == g.ERR_ALIGNMENT
    assert call(C=base + 4, beta=1.0) == g.ERR_ALIGNMENT
    # column-major C/D swaps the operands: ldd then covers M
    col = g.PlanDesc(g.F16, g.F16, g.F16, g.F16, g.F32, 0, 0, 1, 0)
    assert call(desc=col, M=128, ldd=64) == g.ERR_INVALID_ARG
    # 32 tiles of 128 x 256 with 64 splits need 256 MiB of partials
    assert call(M=1024, N=1024, K=4096, lda=4096, ldb=1024, ldd=1024,
                splits=64) == g.ERR_UNSUPPORTED

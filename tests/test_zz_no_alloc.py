"""gemm_run_splitk_noalloc: the split-K entry point for callers that cannot
allocate device memory (hosts that own every byte of the device, or loops
where a cudaMalloc's blocking is unacceptable).  Its partial tiles live in a
fixed device array inside the library; these tests check, through the C ABI,
that two calls in a row reproduce what gemm_run_ex computes on the same
inputs, within the accuracy bound the other parity tests use, and that a
problem needing more scratch than the array holds is refused.

The file is named to be collected last, so that a run stopping at its first
failure has already run every other test."""
import numpy as np
import pytest
import torch

from dense_gemm_15_gb300 import binding as g
from dense_gemm_15_gb300 import inputs
from oracle import check

pytestmark = pytest.mark.gpu

LAYOUT = {False: g.ROW_MAJOR, True: g.COL_MAJOR}


def _existing(prob, A, B, C):
    plan = g.Plan(prob.a_dtype, prob.d_dtype, relu=prob.relu,
                  layout_a=LAYOUT[prob.a_col_major], layout_b=LAYOUT[prob.b_col_major])
    D = torch.empty(prob.M, prob.N, dtype=inputs.TORCH_DTYPE[prob.d_dtype], device="cuda")
    plan.run(A, B, C, D, prob.M, prob.N, prob.K, alpha=prob.alpha, beta=prob.beta)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    return D


def _noalloc(prob, A, B, C, splits, status):
    D = torch.full((prob.M, prob.N), float("nan"), dtype=inputs.TORCH_DTYPE[prob.d_dtype],
                   device="cuda")
    lda = prob.M if prob.a_col_major else prob.K
    ldb = prob.K if prob.b_col_major else prob.N
    st = g.gemm_run_splitk_noalloc(prob.a_dtype, LAYOUT[prob.a_col_major],
                                   LAYOUT[prob.b_col_major], g.ROW_MAJOR, prob.relu,
                                   A, lda, B, ldb, C, prob.N, D, prob.N, prob.M, prob.N, prob.K,
                                   prob.alpha, prob.beta, splits=splits, status=status)
    assert st == g.OK, g.status_string(st)
    torch.cuda.synchronize()
    assert int(status.item()) == g.OK
    return D


@pytest.mark.parametrize("dtype,shape,splits,cols", [
    ("f16", (256, 384, 8192), 8, (False, False)),
    ("bf16", (304, 136, 4160), 5, (True, False)),
    ("f16", (128, 1024, 2048), 3, (False, True)),
])
def test_noalloc_matches_gemm_run_ex_on_two_calls(dtype, shape, splits, cols):
    M, N, K = shape
    prob = inputs.random_problem(M, N, K, dtype=dtype, beta=0.5, alpha=1.5, relu=True,
                                 a_col_major=cols[0], b_col_major=cols[1])
    A, B, C = prob.A.cuda(), prob.B.cuda(), prob.C.cuda()
    ref = inputs.bits(_existing(prob, A, B, C).cpu())
    ref_val = check.decode(ref, prob.d_dtype)
    # tolerance of the parity tests, from the oracle's |A|.|B| and C
    _, absab, c64 = check.reference(prob, inputs.bits)
    tol = check.bound(absab, prob.alpha, prob.beta, c64, prob.d_dtype)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    first = None
    for _ in range(2):
        d = inputs.bits(_noalloc(prob, A, B, C, splits, status).cpu())
        err = np.abs(check.decode(d, prob.d_dtype) - ref_val)
        assert np.all(err <= tol), "max err/tol %.3g" % float(np.max(err / tol))
        if first is None:
            first = d
        else:
            assert np.array_equal(first, d), "second call differs from the first"


def test_noalloc_refuses_more_scratch_than_it_has():
    # 32 tiles of 128 x 256 with 64 splits need 256 MiB of partials
    M, N, K = 1024, 1024, 4096
    A = torch.zeros(M, K, dtype=torch.float16, device="cuda")
    B = torch.zeros(K, N, dtype=torch.float16, device="cuda")
    D = torch.full((M, N), 5.0, dtype=torch.float16, device="cuda")
    st = g.gemm_run_splitk_noalloc("f16", g.ROW_MAJOR, g.ROW_MAJOR, g.ROW_MAJOR, False, A, K,
                                   B, N, None, N, D, N, M, N, K, 1.0, 0.0, splits=64)
    assert st == g.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(D == 5.0)
    assert g.gemm_run_splitk_noalloc("f16", g.ROW_MAJOR, g.ROW_MAJOR, g.ROW_MAJOR, False, A, K,
                                     B, N, None, N, D, N, M, N, K, 1.0, 0.0,
                                     splits=0) == g.ERR_INVALID_ARG

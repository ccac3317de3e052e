"""gemm_run_splitk_noalloc: the split-K entry point for callers that cannot
allocate device memory (hosts that own every byte of the device, or loops
where a cudaMalloc's blocking is unacceptable).  Its partial tiles live in a
fixed device array inside the library.  These tests call it through the C ABI
twice in a row on the same inputs and check both results against the oracle:
bit for bit on small-integer operands (exact fp32 arithmetic), within the
accuracy bound of the other parity tests on random operands, and against the
existing entry point gemm_run_ex.  They cover column-major C/D with every
operand layout, fp8 with per-tensor scales, K == 0, and the refusal of a
problem that needs more scratch than the array holds.

The file is named to be collected last, so that a run stopping at its first
failure has already run every other test."""
import numpy as np
import pytest
import torch

from dense_gemm_15_gb300 import binding as g
from dense_gemm_15_gb300 import inputs
from helpers import assert_bit_exact, assert_matches_oracle

pytestmark = pytest.mark.gpu

LAYOUT = {False: g.ROW_MAJOR, True: g.COL_MAJOR}


def _noalloc(prob, A, B, C, splits, status, col_cd=False):
    """Runs prob through gemm_run_splitk_noalloc; returns D (M x N row-major bits)."""
    dt = inputs.TORCH_DTYPE[prob.d_dtype]
    shape = (prob.N, prob.M) if col_cd else (prob.M, prob.N)
    D = torch.full(shape, float("nan"), dtype=dt, device="cuda")
    lda = prob.M if prob.a_col_major else prob.K
    ldb = prob.K if prob.b_col_major else prob.N
    ldcd = prob.M if col_cd else prob.N
    sa = sb = None
    if prob.a_dtype == "e4m3":
        sa = torch.tensor([prob.scale_a], dtype=torch.float32, device="cuda")
        sb = torch.tensor([prob.scale_b], dtype=torch.float32, device="cuda")
    st = g.gemm_run_splitk_noalloc(prob.a_dtype, LAYOUT[prob.a_col_major],
                                   LAYOUT[prob.b_col_major], LAYOUT[col_cd], prob.relu,
                                   A, lda, B, ldb, C, ldcd, D, ldcd, prob.M, prob.N, prob.K,
                                   prob.alpha, prob.beta, scale_a=sa, scale_b=sb, splits=splits,
                                   status=status)
    assert st == g.OK, g.status_string(st)
    torch.cuda.synchronize()
    assert int(status.item()) == g.OK
    Dh = D.cpu()
    return inputs.bits(Dh.t().contiguous() if col_cd else Dh)


def _operands(prob, col_cd):
    A, B = prob.A.cuda(), prob.B.cuda()
    C = None
    if prob.C is not None:
        C = (prob.C.t().contiguous() if col_cd else prob.C).cuda()
    return A, B, C


def _existing(prob, col_cd):
    """The same problem through gemm_run_ex on a plan."""
    plan = g.Plan(prob.a_dtype, prob.d_dtype, relu=prob.relu,
                  layout_a=LAYOUT[prob.a_col_major], layout_b=LAYOUT[prob.b_col_major],
                  layout_cd=LAYOUT[col_cd])
    A, B, C = _operands(prob, col_cd)
    dt = inputs.TORCH_DTYPE[prob.d_dtype]
    D = torch.empty((prob.N, prob.M) if col_cd else (prob.M, prob.N), dtype=dt, device="cuda")
    sa = sb = None
    if prob.a_dtype == "e4m3":
        sa = torch.tensor([prob.scale_a], dtype=torch.float32, device="cuda")
        sb = torch.tensor([prob.scale_b], dtype=torch.float32, device="cuda")
    plan.run(A, B, C, D, prob.M, prob.N, prob.K, alpha=prob.alpha, beta=prob.beta,
             scale_a=sa, scale_b=sb)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    Dh = D.cpu()
    return inputs.bits(Dh.t().contiguous() if col_cd else Dh)


CASES = [
    # dtype, (M, N, K), splits, (A col-major, B col-major), C/D col-major
    ("f16", (256, 384, 8192), 8, (False, False), False),
    ("bf16", (304, 136, 4160), 5, (True, False), False),
    ("f16", (128, 1024, 2048), 3, (False, True), False),
    ("bf16", (264, 392, 2112), 4, (False, False), True),
    ("f16", (200, 520, 4096), 6, (True, True), True),
    ("bf16", (392, 136, 1024), 2, (False, True), True),
    ("e4m3", (264, 528, 4224), 7, (False, False), False),
    ("e4m3", (256, 272, 2048), 3, (False, False), True),
]


@pytest.mark.parametrize("dtype,shape,splits,cols,col_cd", CASES)
def test_noalloc_bit_exact_on_two_calls(dtype, shape, splits, cols, col_cd):
    """Small-integer operands: both calls equal the oracle's rounded result
    bit for bit (fp8 with scales 1/2 and 1/4, bf16 output)."""
    M, N, K = shape
    kw = dict(beta=0.0, scale_a=0.5, scale_b=0.25) if dtype == "e4m3" else dict(beta=0.5)
    prob = inputs.integer_problem(M, N, K, dtype=dtype, act="relu", a_col_major=cols[0],
                                  b_col_major=cols[1], **kw)
    A, B, C = _operands(prob, col_cd)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        assert_bit_exact(prob, _noalloc(prob, A, B, C, splits, status, col_cd))


@pytest.mark.parametrize("dtype,shape,splits,cols,col_cd", CASES[:3] + CASES[4:5] + CASES[7:])
def test_noalloc_matches_oracle_and_gemm_run_ex_on_two_calls(dtype, shape, splits, cols, col_cd):
    """Random operands: both calls within the oracle's bound and bit-equal to
    each other; the existing entry point gemm_run_ex within the same bound."""
    M, N, K = shape
    kw = dict(beta=0.0, scale_a=0.37, scale_b=1.7) if dtype == "e4m3" else dict(beta=0.5)
    prob = inputs.random_problem(M, N, K, dtype=dtype, alpha=1.5, relu=True,
                                 a_col_major=cols[0], b_col_major=cols[1], **kw)
    A, B, C = _operands(prob, col_cd)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    first = None
    for _ in range(2):
        d = _noalloc(prob, A, B, C, splits, status, col_cd)
        assert_matches_oracle(prob, d)
        if first is None:
            first = d
        else:
            assert np.array_equal(first, d), "second call differs from the first"
    assert_matches_oracle(prob, _existing(prob, col_cd))


def test_noalloc_k_zero_is_act_of_beta_c():
    """K == 0 launches the reduction alone: D = relu(beta * C), bit-exact."""
    prob = inputs.integer_problem(70, 136, 0, dtype="f16", act="relu", beta=0.5)
    prob.A = torch.empty(70, 0, dtype=torch.float16)
    prob.B = torch.empty(0, 136, dtype=torch.float16)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    dummy = torch.empty(8, dtype=torch.float16, device="cuda")
    for _ in range(2):
        assert_bit_exact(prob, _noalloc(prob, dummy, dummy, prob.C.cuda(), 3, status))


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

"""Parity of the sm_103a GEMM against the CPU oracle, through the C ABI.

Bit-exact where the result is exact (the pages' all-ones examples, identity,
zero and ReLU cases); otherwise within the accuracy bound
|D - D_ref| <= 1e-2 |alpha| (|A|.|B|) + 1e-3 (+ output rounding of beta*C)."""
import numpy as np
import pytest
import torch

from dense_gemm_15_gb300 import binding as g
from dense_gemm_15_gb300 import inputs
from conftest import read_golden
from helpers import (assert_matches_oracle, assert_windows_match_oracle, band_windows, plan_for,
                     run_gpu)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fixture", ["all_ones_128.txt", "all_ones_1024.txt"])
def test_all_ones_examples_bit_exact(fixture):
    gd = read_golden(fixture)
    n = int(gd["M"][0][0])
    prob = inputs.Problem("ones", inputs.ones((n, n), "f16"), inputs.ones((n, n), "f16"),
                          inputs.ones((n, n), "f16"), n, n, n, alpha=1.0, beta=1.0)
    d = run_gpu(plan_for(prob), prob)
    assert np.all(d == int(gd["expect_bits_all"][0][0], 16))


def test_uniform_1024_matches_oracle():
    prob = inputs.config1("b")
    assert_matches_oracle(prob, run_gpu(plan_for(prob), prob))


def test_alpha_beta_relu_hand_example():
    gd = read_golden("alpha_beta_relu_2x2.txt")
    # embed the 2x2 example in an 8x8 problem (16-byte aligned rows)
    A = torch.zeros(8, 8, dtype=torch.float16)
    B = torch.zeros(8, 8, dtype=torch.float16)
    C = torch.zeros(8, 8, dtype=torch.float16)
    A[:2, :2] = torch.tensor([float(v) for v in gd["A"][0]]).reshape(2, 2)
    B[:2, :2] = torch.tensor([float(v) for v in gd["B"][0]]).reshape(2, 2)
    C[:2, :2] = torch.tensor([float(v) for v in gd["C"][0]]).reshape(2, 2)
    prob = inputs.Problem("hand", A, B, C, 8, 8, 8, alpha=1.5, beta=0.5, relu=True)
    d = run_gpu(plan_for(prob), prob).view(np.float16).astype(np.float64)
    expect = np.array([float(v) for v in gd["expect"][0]]).reshape(2, 2)
    assert np.array_equal(d[:2, :2], expect)
    assert np.all(d[2:, :] == 0) and np.all(d[:, 2:] == 0)


@pytest.mark.parametrize("shape", [(128, 64, 256), (32, 256, 128)])
def test_plan_reuse_extra_shapes(shape):
    """One plan (alpha 1.5, beta 0.5, ReLU) reused across the extra shapes."""
    M, N, K = shape
    plan = None
    for (m, n, k) in [(M, N, K), (4096 // 16, 256, 512)]:
        prob = inputs.config2(m, n, k)
        plan = plan or plan_for(prob)
        assert_matches_oracle(prob, run_gpu(plan, prob))


def test_identity_and_zero_bit_exact():
    K = N = 256
    A = inputs.uniform((300, K), -4, 4, "f16", 90, 1)
    eye = torch.eye(K, dtype=torch.float16)
    prob = inputs.Problem("identity", A, eye, None, 300, N, K)
    assert np.array_equal(run_gpu(plan_for(prob), prob), inputs.bits(A))
    C = inputs.uniform((300, N), -4, 4, "f16", 90, 2)
    zero = inputs.Problem("zeroA", torch.zeros(300, K, dtype=torch.float16), eye, C,
                          300, N, K, alpha=1.0, beta=0.5)
    want = (C.to(torch.float64) * 0.5).to(torch.float16)
    assert np.array_equal(run_gpu(plan_for(zero), zero), inputs.bits(want))


def test_relu_of_negative_is_zero():
    A = -torch.ones(256, 64, dtype=torch.float16)
    B = torch.ones(64, 512, dtype=torch.float16)
    prob = inputs.Problem("neg", A, B, None, 256, 512, 64, relu=True)
    assert np.all(run_gpu(plan_for(prob), prob) == 0)


@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (7, 24, 40), (129, 264, 72), (200, 304, 136),
                                   (333, 520, 1000), (128, 256, 64), (256, 512, 8)])
def test_ragged_shapes(M, N, K):
    prob = inputs.random_problem(M, N, K, beta=1.0, alpha=1.0)
    assert_matches_oracle(prob, run_gpu(plan_for(prob), prob))


@pytest.mark.parametrize("a_col,b_col", [(False, False), (True, False), (False, True), (True, True)])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_layouts_and_dtypes(a_col, b_col, dtype):
    prob = inputs.random_problem(264, 392, 200, dtype=dtype, beta=0.5, alpha=1.5, relu=True,
                                 a_col_major=a_col, b_col_major=b_col)
    assert_matches_oracle(prob, run_gpu(plan_for(prob), prob))


def test_beta_zero_never_reads_c():
    prob = inputs.random_problem(130, 264, 96, beta=0.0)
    plan = plan_for(prob)
    nan_c = torch.full((prob.M, prob.N), float("nan"), dtype=torch.float16, device="cuda")
    D = torch.empty_like(nan_c)
    plan.run(prob.A.cuda(), prob.B.cuda(), nan_c, D, prob.M, prob.N, prob.K, alpha=1.0, beta=0.0)
    torch.cuda.synchronize()
    assert torch.isfinite(D).all()
    assert_matches_oracle(prob, inputs.bits(D.cpu()))


def test_config2_full_size_sampled_rows():
    prob = inputs.config2()
    d = run_gpu(plan_for(prob), prob)
    assert_windows_match_oracle(prob, d, band_windows(prob.M, band=256, span=8))
    strong = inputs.config2(strong=True)
    d = run_gpu(plan_for(strong), strong)
    assert_matches_oracle(strong, d, rows=(4096 - 64, 4096))


def test_alpha_zero_gives_rounded_beta_c():
    """alpha = 0: the product term vanishes, D = rne(beta * C) bit-exactly."""
    prob = inputs.random_problem(200, 264, 136, alpha=0.0, beta=0.5)
    want = (prob.C.to(torch.float64) * 0.5).to(torch.float16)
    assert np.array_equal(run_gpu(plan_for(prob), prob), inputs.bits(want))


@pytest.mark.parametrize("K", [1, 7, 63, 64, 65, 127, 129])
def test_k_around_one_k_block(K):
    """K from 1 to just past two k-blocks of 64, with A and B padded to a
    16-byte leading dimension (the K tail is zero-filled by the TMA)."""
    M, N = 130, 264
    prob = inputs.random_problem(M, N, K, beta=1.0, relu=True)
    lda = (K + 7) // 8 * 8
    A = torch.zeros(M, lda, dtype=torch.float16)
    A[:, :K] = prob.A
    plan = plan_for(prob)
    D = torch.empty(M, N, dtype=torch.float16, device="cuda")
    plan.run(A.cuda(), prob.B.cuda(), prob.C.cuda(), D, M, N, K, alpha=1.0, beta=1.0, lda=lda)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    assert_matches_oracle(prob, inputs.bits(D.cpu()))

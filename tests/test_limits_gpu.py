"""Size limits on the GPU, bit-exact on sampled rows: an output of more than
2^31 elements (64-bit addressing of C, D and the epilogue's stores) and a K
of 2^20 (split-K over many k-blocks).  Small-integer operands keep every sum
exact in fp32, so the sampled rows must equal the oracle's rounded result."""
import numpy as np
import pytest
import torch

from dense_gemm_15_gb300 import binding as g
from dense_gemm_15_gb300 import inputs
from helpers import assert_bit_exact, band_windows, row_subproblem

pytestmark = pytest.mark.gpu


def _windows_bit_exact(prob, D, windows):
    idx = np.concatenate([np.arange(a, b) for a, b in windows])
    rows = D[torch.as_tensor(idx, device=D.device)].cpu()
    assert_bit_exact(row_subproblem(prob, idx), inputs.bits(rows))


def test_output_of_more_than_two_to_the_31_elements():
    """65536 x 40960 = 2.7e9 outputs (5.4 GB of bf16), K = 64: rows in every
    4096-row band and the last rows."""
    M, N, K = 65536, 40960, 64
    assert M * N > 2 ** 31
    prob = inputs.integer_problem(M, N, K, dtype="bf16", alpha=1.0, beta=0.0, act="relu")
    plan = g.Plan("bf16", "bf16", relu=True)
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    plan.run(prob.A.cuda(), prob.B.cuda(), None, D, M, N, K)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    _windows_bit_exact(prob, D, band_windows(M, band=4096, span=2))
    del D
    torch.cuda.empty_cache()


def test_k_of_two_to_the_20():
    """256 x 256 x 1048576 (split-K over 16384 k-blocks): |D| <= 4 * 2^20 < 2^24."""
    M, N, K = 256, 256, 1 << 20
    prob = inputs.integer_problem(M, N, K, dtype="bf16", alpha=1.0, beta=0.0, act="linear")
    plan = g.Plan("bf16", "bf16")
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    plan.run(prob.A.cuda(), prob.B.cuda(), None, D, M, N, K)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    _windows_bit_exact(prob, D, band_windows(M, band=128, span=4))

"""Batched GEMM (batch_count / batch_stride of the kwkr.cn blog "CUTLASS
Python接口", section 6.3) against the oracle, entry by entry, through the C ABI."""
import numpy as np
import pytest
import torch

from dense_gemm_15_gb300 import binding as g
from dense_gemm_15_gb300 import inputs
from helpers import assert_matches_oracle, plan_for

pytestmark = pytest.mark.gpu


def _stack(tensors, stride):
    """One flat buffer holding tensor b at element b * stride; the gaps are NaN."""
    n = tensors[0].numel()
    flat = torch.full((stride * (len(tensors) - 1) + n,), float("nan"), dtype=tensors[0].dtype)
    for b, t in enumerate(tensors):
        flat[b * stride:b * stride + n] = t.reshape(-1)
    return flat


@pytest.mark.parametrize("dtype,a_col,b_col,share_b,pad", [
    ("f16", False, False, False, 0),
    ("f16", False, False, True, 24),
    ("bf16", True, False, False, 8),
    ("bf16", False, True, True, 0),
    ("f16", True, True, False, 40),
    ("e4m3", False, False, False, 0),
    ("e4m3", False, True, True, 16),
])
def test_batched_matches_oracle_per_entry(dtype, a_col, b_col, share_b, pad):
    batch, M, N, K = 4, 200, 264, 136
    if dtype == "e4m3":
        N, K = 272, 144  # one-byte rows: N and K multiples of 16
    probs = [inputs.random_problem(M, N, K, dtype=dtype, alpha=1.5, beta=0.5, relu=True,
                                   a_col_major=a_col, b_col_major=b_col, seed=b)
             for b in range(batch)]
    if share_b:
        for p in probs:
            p.B = probs[0].B
    sa, sb, sc, sd = M * K + pad, 0 if share_b else K * N + pad, M * N + pad, M * N + pad
    A = _stack([p.A for p in probs], sa).cuda()
    B = (probs[0].B.reshape(-1) if share_b else _stack([p.B for p in probs], sb)).cuda()
    C = _stack([p.C for p in probs], sc).cuda()
    D = torch.full((sd * (batch - 1) + M * N,), float("nan"), dtype=probs[0].C.dtype,
                   device="cuda")
    plan = plan_for(probs[0])
    plan.batched(A, B, C, D, M, N, K, batch, sa, sb, sc, sd, alpha=1.5, beta=0.5)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    cfg = plan.last_config()
    assert cfg["tiles"] == batch * 2 * 2  # 200 rows -> 2 blocks of 128, 264 cols -> 2 of 256
    Dh = D.cpu()
    for b, p in enumerate(probs):
        assert_matches_oracle(p, inputs.bits(Dh[b * sd:b * sd + M * N].reshape(M, N)))
        if pad and b + 1 < batch:
            assert torch.isnan(Dh[b * sd + M * N:(b + 1) * sd]).all(), "wrote between entries"


@pytest.mark.parametrize("cta_group", [1, 2])
def test_batched_tile_shapes(cta_group):
    """The same batch on single-SM and on SM-pair tiles."""
    batch, M, N, K = 6, 392, 520, 264
    probs = [inputs.random_problem(M, N, K, dtype="bf16", beta=1.0, act="tanh", seed=b)
             for b in range(batch)]
    A = torch.stack([p.A for p in probs]).cuda()
    B = torch.stack([p.B for p in probs]).cuda()
    C = torch.stack([p.C for p in probs]).cuda()
    D = torch.empty(batch, M, N, dtype=torch.bfloat16, device="cuda")
    plan = g.Plan("bf16", epilogue="tanh").set(g.OPT_CTA_GROUP, cta_group)
    plan.batched(A, B, C, D, M, N, K, batch, M * K, K * N, M * N, M * N, beta=1.0)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    assert plan.last_config()["cta_group"] == cta_group
    Dh = D.cpu()
    for b, p in enumerate(probs):
        assert_matches_oracle(p, inputs.bits(Dh[b]))


def test_batched_argument_errors():
    M, N, K = 64, 128, 64
    p = inputs.random_problem(M, N, K, beta=1.0)
    plan = plan_for(p)
    A, B, C = p.A.cuda(), p.B.cuda(), p.C.cuda()
    D = torch.empty(M, N, dtype=torch.float16, device="cuda")
    run = lambda *strides, batch=1: g.gemm_run_batched(plan.handle, A, 0, strides[0], B, 0,
                                                       strides[1], C, 0, strides[2], D, 0,
                                                       strides[3], M, N, K, batch, 1.0, 1.0)
    assert run(4, 0, 0, 0) == g.ERR_ALIGNMENT        # 8 bytes
    assert run(0, 0, 0, 0, batch=-1) == g.ERR_INVALID_ARG
    assert run(-8, 0, 0, 0) == g.ERR_INVALID_ARG
    assert run(0, 0, 0, 0, batch=0) == g.OK            # nothing to do
    assert run(0, 0, 0, 0) == g.OK                     # one entry
    torch.cuda.synchronize()
    assert_matches_oracle(p, inputs.bits(D.cpu()))


def test_repeated_calls_reuse_and_refresh_the_problem_table():
    """A call with the same problems reuses the device table (the data at the
    same pointers may change); a call with other pointers rebuilds it."""
    batch, M, N, K = 3, 136, 256, 64
    probs = [inputs.random_problem(M, N, K, seed=b) for b in range(batch)]
    A = torch.stack([p.A for p in probs]).cuda()
    B = torch.stack([p.B for p in probs]).cuda()
    D = torch.empty(batch, M, N, dtype=torch.float16, device="cuda")
    plan = plan_for(probs[0])
    args = (M, N, K, batch, M * K, K * N, 0, M * N)
    plan.batched(A, B, None, D, *args)
    # same pointers, new contents
    probs2 = [inputs.random_problem(M, N, K, seed=10 + b) for b in range(batch)]
    A.copy_(torch.stack([p.A for p in probs2]))
    plan.batched(A, B, None, D, *args)
    torch.cuda.synchronize()
    Dh = D.cpu()
    for b in range(batch):
        probs2[b].B = probs[b].B
        assert_matches_oracle(probs2[b], inputs.bits(Dh[b]))
    # other pointers: every entry uses the first B
    D2 = torch.empty_like(D)
    plan.batched(A, B, None, D2, M, N, K, batch, M * K, 0, 0, M * N)
    torch.cuda.synchronize()
    Dh = D2.cpu()
    for b in range(batch):
        probs2[b].B = probs[0].B
        assert_matches_oracle(probs2[b], inputs.bits(Dh[b]))
    assert plan.query_error() == g.OK

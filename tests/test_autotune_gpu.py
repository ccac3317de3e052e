"""Autotuning (kwkr.cn blog "CUTLASS Python接口", section 6.2: profile the
configurations for a problem size and fix the fastest) through the C ABI."""
import pytest
import torch

from dense_gemm_15_gb300 import binding as g
from dense_gemm_15_gb300 import inputs
from helpers import assert_matches_oracle, plan_for

pytestmark = pytest.mark.gpu

KEYS = ("schedule", "cta_group", "tile_n", "splits")


def _dev(prob):
    A, B = prob.A.cuda(), prob.B.cuda()
    C = prob.C.cuda() if prob.C is not None else None
    D = torch.empty(prob.M, prob.N, dtype=inputs.TORCH_DTYPE[prob.d_dtype], device="cuda")
    return A, B, C, D


@pytest.mark.parametrize("dtype,n_cands", [("f16", 16), ("e4m3", 12)])
def test_autotune_keeps_the_fastest_and_later_runs_use_it(dtype, n_cands):
    prob = inputs.random_problem(1536, 1536, 4096, dtype=dtype, alpha=1.5,
                                 beta=0.5 if dtype == "f16" else 0.0, relu=True)
    plan = plan_for(prob)
    A, B, C, D = _dev(prob)
    res = plan.autotune(A, B, C, D, prob.M, prob.N, prob.K, prob.alpha, prob.beta, iterations=3)
    assert len(res) == n_cands
    assert all(r["status"] == g.OK and r["us"] > 0 for r in res)
    times = [r["us"] for r in res]
    assert times == sorted(times)
    assert {r["config"]["schedule"] for r in res} == {g.SCHED_DP, g.SCHED_SK, g.SCHED_SPLIT}
    best = res[0]["config"]
    # D holds the chosen configuration's result, and so does a later run
    torch.cuda.synchronize()
    assert_matches_oracle(prob, inputs.bits(D.cpu()))
    assert all(plan.last_config()[k] == best[k] for k in KEYS)
    D.fill_(float("nan"))
    plan.run(A, B, C, D, prob.M, prob.N, prob.K, alpha=prob.alpha, beta=prob.beta)
    torch.cuda.synchronize()
    assert all(plan.last_config()[k] == best[k] for k in KEYS)
    assert_matches_oracle(prob, inputs.bits(D.cpu()))


def test_explicit_options_win_and_forgetting_restores_the_heuristic():
    prob = inputs.random_problem(1024, 2048, 2048, beta=1.0)
    A, B, C, D = _dev(prob)
    fresh = plan_for(prob)
    fresh.run(A, B, C, D, prob.M, prob.N, prob.K, alpha=1.0, beta=1.0)
    heuristic = fresh.last_config()
    plan = plan_for(prob)
    best = plan.autotune(A, B, C, D, prob.M, prob.N, prob.K, 1.0, 1.0, iterations=2)[0]["config"]
    other = g.SCHED_DP if best["schedule"] != g.SCHED_DP else g.SCHED_SPLIT
    plan.set(g.OPT_SCHEDULE, other)
    plan.run(A, B, C, D, prob.M, prob.N, prob.K, alpha=1.0, beta=1.0)
    assert plan.last_config()["schedule"] == other
    plan.set(g.OPT_SCHEDULE, g.SCHED_AUTO)
    assert g.gemm_plan_forget_tuning(plan.handle) == g.OK
    plan.run(A, B, C, D, prob.M, prob.N, prob.K, alpha=1.0, beta=1.0)
    torch.cuda.synchronize()
    assert all(plan.last_config()[k] == heuristic[k] for k in KEYS)
    assert_matches_oracle(prob, inputs.bits(D.cpu()))


def test_autotune_argument_errors():
    prob = inputs.random_problem(64, 128, 64)
    plan = plan_for(prob)
    A, B, C, D = _dev(prob)
    st, _ = g.gemm_plan_autotune(plan.handle, A, B, None, D, 64, 128, 64, iterations=0)
    assert st == g.ERR_INVALID_ARG
    st, res = g.gemm_plan_autotune(plan.handle, A, B, None, D, 64, 128, 0)
    assert st == g.OK and res == []
    st, _ = g.gemm_plan_autotune(plan.handle, A, B, None, D, 64, 128, 64,
                                 bias=torch.zeros(136, dtype=torch.float16, device="cuda")[4:])
    assert st == g.ERR_ALIGNMENT


def test_autotune_includes_swap_ab_for_a_short_side():
    """A decode-size problem (M = 32) adds the three swap-AB schedules to the
    candidates; whichever wins, later runs of the shape reproduce it."""
    prob = inputs.random_problem(32, 4096, 4096, dtype="bf16")
    plan = plan_for(prob)
    A, B, C, D = _dev(prob)
    res = plan.autotune(A, B, C, D, prob.M, prob.N, prob.K, 1.0, 0.0, iterations=2)
    assert len(res) == 19
    assert sum(r["config"]["swap_ab"] for r in res) == 3
    best = res[0]["config"]
    torch.cuda.synchronize()
    assert_matches_oracle(prob, inputs.bits(D.cpu()))
    plan.run(A, B, C, D, prob.M, prob.N, prob.K)
    assert all(plan.last_config()[k] == best[k] for k in KEYS + ("swap_ab",))

"""Shared helpers of the GPU parity tests: run a seeded problem through the
C ABI and compare it with the oracle on the same inputs."""
import numpy as np
import torch

from dense_gemm_15_gb300 import binding as g
from dense_gemm_15_gb300 import inputs
from oracle import check

LAYOUT = {False: g.ROW_MAJOR, True: g.COL_MAJOR}


def plan_for(prob, **opts):
    plan = g.Plan(prob.a_dtype, prob.d_dtype, epilogue=prob.act,
                  layout_a=LAYOUT[prob.a_col_major], layout_b=LAYOUT[prob.b_col_major])
    for k, v in opts.items():
        plan.set(getattr(g, "OPT_" + k.upper()), v)
    return plan


def run_gpu(plan, prob, device="cuda", d_init=None, scales_dev=None):
    """Runs prob on the GPU through the C ABI; returns D's stored bits (numpy)."""
    A = prob.A.to(device)
    B = prob.B.to(device)
    C = prob.C.to(device) if prob.C is not None else None
    if d_init is not None:
        D = d_init.to(device).clone()
    else:
        D = torch.empty((prob.M, prob.N), dtype=inputs.TORCH_DTYPE[prob.d_dtype], device=device)
    sa = sb = None
    if prob.a_dtype == "e4m3" and (prob.scale_a != 1.0 or prob.scale_b != 1.0 or scales_dev):
        sa = torch.tensor([prob.scale_a], dtype=torch.float32, device=device)
        sb = torch.tensor([prob.scale_b], dtype=torch.float32, device=device)
    plan.run(A, B, C, D, prob.M, prob.N, prob.K, alpha=prob.alpha, beta=prob.beta,
             scale_a=sa, scale_b=sb)
    torch.cuda.synchronize()
    status = plan.query_error()
    assert status == g.OK, g.status_string(status)
    return inputs.bits(D.cpu())


def assert_matches_oracle(prob, d_bits, rows=None):
    d_ref, absab, c64 = check.reference(prob, inputs.bits, rows=rows)
    r0, r1 = (0, prob.M) if rows is None else rows
    ok, worst, idx, nbad = check.compare(d_bits[r0:r1], prob.d_dtype, d_ref, absab, c64, prob)
    assert ok, "%s: %d elements out of tolerance, worst ratio %.3g at %s" % (
        prob.name, nbad, worst, idx)
    return worst


def sample_rows(M, count=3, span=64, seed=0):
    """A few row windows spread over [0, M), including the last rows."""
    if M <= span * count:
        return [(0, M)]
    rng = np.random.default_rng(seed)
    starts = sorted(set([0, M - span] + [int(x) for x in rng.integers(0, M - span, count - 2)]))
    return [(s, s + span) for s in starts]

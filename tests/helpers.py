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


def oracle_bits(prob):
    """The oracle's D rounded once to the output type (nearest even): the
    expected stored bits of a problem whose arithmetic is exact in fp32."""
    import oracle
    a, b = inputs.bits(prob.A), inputs.bits(prob.B)
    c = inputs.bits(prob.C) if prob.C is not None and prob.beta != 0.0 else None
    bias = inputs.bits(prob.bias) if prob.bias is not None else None
    aux = inputs.bits(prob.aux) if prob.aux_op else None
    d = oracle.gemm(a, prob.a_dtype, b, prob.b_dtype, c, prob.c_dtype, alpha=prob.alpha,
                    beta=prob.beta, act=prob.act, bias=bias, bias_dtype=prob.d_dtype,
                    aux=aux, aux_dtype=prob.d_dtype, aux_op=prob.aux_op,
                    scale_a=prob.scale_a, scale_b=prob.scale_b,
                    a_col_major=prob.a_col_major, b_col_major=prob.b_col_major)
    return oracle.round_to(d, prob.d_dtype)


def assert_bit_exact(prob, d_bits, want=None):
    want = oracle_bits(prob) if want is None else want
    assert d_bits.shape == want.shape
    bad = np.argwhere(d_bits != want)
    assert bad.size == 0, "%s: %d elements differ from the oracle, first at %s (%#06x vs %#06x)" % (
        prob.name, len(bad), tuple(bad[0]), int(d_bits[tuple(bad[0])]), int(want[tuple(bad[0])]))


def band_windows(M, band=256, span=8, seed=0):
    """One window of `span` rows at a seeded offset inside every `band`-row
    band of [0, M), plus the last `span` rows: every M-tile band of the
    kernels (128 or 256 rows) is sampled."""
    rng = np.random.default_rng([seed, M, band])
    wins = set()
    for b0 in range(0, M, band):
        hi = min(M, b0 + band)
        s = b0 + int(rng.integers(0, max(1, hi - b0 - span + 1)))
        wins.add((s, min(hi, s + span)))
    wins.add((max(0, M - span), M))
    return sorted(wins)


def row_subproblem(prob, idx):
    """The problem restricted to rows `idx` of A, C, Z and D (a row of D
    depends only on the same row of A, C and Z)."""
    import copy
    idx = torch.as_tensor(np.asarray(idx, dtype=np.int64))
    sub = copy.copy(prob)
    # rows are gathered on the stored bytes (torch has no CPU indexing for fp8)
    a = prob.A.view(torch.uint8) if prob.A.element_size() == 1 else prob.A
    a = (a[:, idx] if prob.a_col_major else a[idx]).contiguous()
    sub.A = a.view(prob.A.dtype) if prob.A.element_size() == 1 else a
    sub.C = prob.C[idx].contiguous() if prob.C is not None else None
    if getattr(prob, "aux", None) is not None:
        sub.aux = prob.aux[idx].contiguous()
    sub.M = int(idx.numel())
    sub.name = prob.name + "[rows]"
    return sub


def assert_windows_match_oracle(prob, d_bits, windows):
    """Compares the rows of `windows` against one oracle call on those rows."""
    idx = np.concatenate([np.arange(a, b) for a, b in windows])
    sub = row_subproblem(prob, idx)
    return assert_matches_oracle(sub, np.ascontiguousarray(d_bits[idx]))

"""Richer fused epilogues against the oracle, through the C ABI: a per-column
bias (kwkr.cn blog "CUTLASS Python接口", section 5.2, LinearCombinationBiasReLU)
and sigmoid / tanh activations ("Generating State-of-the-Art GEMMs with
TorchInductor's CuteDSL backend", roadmap section)."""
import numpy as np
import pytest
import torch

from dense_gemm_15_gb300 import binding as g
from dense_gemm_15_gb300 import inputs
from helpers import LAYOUT, assert_matches_oracle

pytestmark = pytest.mark.gpu


def _plan(prob, layout_cd=g.ROW_MAJOR, **opts):
    plan = g.Plan(prob.a_dtype, prob.d_dtype, epilogue=prob.act,
                  layout_a=LAYOUT[prob.a_col_major], layout_b=LAYOUT[prob.b_col_major],
                  layout_cd=layout_cd)
    for k, v in opts.items():
        plan.set(getattr(g, "OPT_" + k.upper()), v)
    return plan


def _run(plan, prob, ldd=None, col_major_cd=False):
    """Runs prob (bias included) and returns D as an M x N row-major bit array."""
    A, B = prob.A.cuda(), prob.B.cuda()
    C = prob.C.cuda() if prob.C is not None else None
    bias = prob.bias.cuda() if prob.bias is not None else None
    dt = inputs.TORCH_DTYPE[prob.d_dtype]
    if col_major_cd:
        C = C.t().contiguous() if C is not None else None  # storage N x M
        D = torch.full((prob.N, prob.M), float("nan"), dtype=dt, device="cuda")
    else:
        D = torch.full((prob.M, ldd or prob.N), float("nan"), dtype=dt, device="cuda")
    sa = sb = None
    if prob.a_dtype == "e4m3":
        sa = torch.tensor([prob.scale_a], dtype=torch.float32, device="cuda")
        sb = torch.tensor([prob.scale_b], dtype=torch.float32, device="cuda")
    st = g.gemm_run_args(plan.handle, A, B, C, D, prob.M, prob.N, prob.K, prob.alpha,
                         prob.beta, ldd=ldd or 0, scale_a=sa, scale_b=sb, bias=bias)
    assert st == g.OK, g.status_string(st)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    Dh = D.cpu()
    if col_major_cd:
        Dh = Dh.t().contiguous()
    else:
        if ldd:
            assert torch.isnan(Dh[:, prob.N:]).all(), "wrote past N"
        Dh = Dh[:, :prob.N].contiguous()
    return inputs.bits(Dh)


@pytest.mark.parametrize("act", ["linear", "relu", "sigmoid", "tanh"])
@pytest.mark.parametrize("bias", [False, True])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_activation_and_bias(act, bias, dtype):
    prob = inputs.random_problem(520, 392, 1096, dtype=dtype, alpha=0.25, beta=0.5,
                                 act=act, bias=bias)
    assert_matches_oracle(prob, _run(_plan(prob), prob))


@pytest.mark.parametrize("act", ["sigmoid", "tanh"])
@pytest.mark.parametrize("sched", [g.SCHED_SK, g.SCHED_SPLIT])
@pytest.mark.parametrize("M", [24, 96])
def test_activations_on_swap_ab_tiles(act, sched, M):
    """Sigmoid and tanh in the transposed (swap-AB) epilogue, with C and a
    bias that runs along the computed rows, on random operands."""
    prob = inputs.random_problem(M, 1160, 2048, dtype="bf16", alpha=0.5, beta=0.5, act=act,
                                 bias=True)
    plan = _plan(prob, schedule=sched, swap_ab=2)
    d = _run(plan, prob)
    assert plan.last_config()["swap_ab"] == 1
    assert_matches_oracle(prob, d)


@pytest.mark.parametrize("sched", [g.SCHED_DP, g.SCHED_SK, g.SCHED_SPLIT])
@pytest.mark.parametrize("col_major_cd", [False, True])
def test_bias_under_every_schedule_and_output_layout(sched, col_major_cd):
    """The bias runs along the computed rows when column-major C/D make the
    kernel compute D^T; split-K adds it in the reduction kernel."""
    prob = inputs.random_problem(296, 264, 2048, dtype="bf16", alpha=1.5, beta=-0.5,
                                 act="relu", bias=True)
    plan = _plan(prob, layout_cd=LAYOUT[col_major_cd], schedule=sched)
    d = _run(plan, prob, col_major_cd=col_major_cd)
    assert plan.last_config()["schedule"] == sched
    assert_matches_oracle(prob, d)


def test_bias_relu_example_shape():
    """Section 5.2's example: M, N, K = 512, 1024, 768, fp16, alpha 1, beta 0,
    bias of length N, ReLU."""
    prob = inputs.random_problem(512, 1024, 768, act="relu", bias=True)
    assert_matches_oracle(prob, _run(_plan(prob), prob))


def test_bias_with_ragged_n_and_padded_ld():
    """N = 131 ends inside a 16-byte group of the bias and of D; B, C and D
    have the padded leading dimension 136."""
    prob = inputs.random_problem(75, 131, 200, beta=1.0, act="tanh", bias=True)
    B = torch.zeros(200, 136, dtype=torch.float16)
    B[:, :131] = prob.B
    C = torch.zeros(75, 136, dtype=torch.float16)
    C[:, :131] = prob.C
    plan = _plan(prob)
    D = torch.full((75, 136), float("nan"), dtype=torch.float16, device="cuda")
    st = g.gemm_run_args(plan.handle, prob.A.cuda(), B.cuda(), C.cuda(), D, 75, 131, 200, 1.0,
                         1.0, ldb=136, ldc=136, ldd=136, bias=prob.bias.cuda())
    assert st == g.OK
    torch.cuda.synchronize()
    Dh = D.cpu()
    assert torch.isnan(Dh[:, 131:]).all()
    assert_matches_oracle(prob, inputs.bits(Dh[:, :131].contiguous()))


def test_bias_with_k_zero_is_act_of_beta_c_plus_bias():
    prob = inputs.random_problem(40, 72, 0, beta=0.75, act="sigmoid", bias=True)
    prob.A = torch.empty(40, 0, dtype=torch.float16)
    prob.B = torch.empty(0, 72, dtype=torch.float16)
    assert_matches_oracle(prob, _run(_plan(prob), prob))


def test_e4m3_with_bias_and_scales():
    prob = inputs.random_problem(264, 512, 1024, dtype="e4m3", alpha=1.0, beta=0.0,
                                 act="relu", bias=True, scale_a=0.5, scale_b=0.25)
    assert_matches_oracle(prob, _run(_plan(prob), prob))


def test_misaligned_bias_is_rejected():
    prob = inputs.random_problem(64, 128, 64, act="relu", bias=True)
    plan = _plan(prob)
    A, B = prob.A.cuda(), prob.B.cuda()
    D = torch.empty(64, 128, dtype=torch.float16, device="cuda")
    bias = torch.zeros(136, dtype=torch.float16, device="cuda")[4:]  # 8-byte offset
    st = g.gemm_run_args(plan.handle, A, B, None, D, 64, 128, 64, 1.0, 0.0, bias=bias)
    assert st == g.ERR_ALIGNMENT


def _run_aux(plan, prob, col_major_cd=False):
    A, B = prob.A.cuda(), prob.B.cuda()
    C = prob.C.cuda() if prob.C is not None else None
    Z = prob.aux.cuda()
    bias = prob.bias.cuda() if prob.bias is not None else None
    dt = inputs.TORCH_DTYPE[prob.d_dtype]
    if col_major_cd:
        C = C.t().contiguous() if C is not None else None
        Z = Z.t().contiguous()
        D = torch.full((prob.N, prob.M), float("nan"), dtype=dt, device="cuda")
    else:
        D = torch.full((prob.M, prob.N), float("nan"), dtype=dt, device="cuda")
    st = g.gemm_run_args(plan.handle, A, B, C, D, prob.M, prob.N, prob.K, prob.alpha,
                         prob.beta, bias=bias, aux=Z, aux_op=prob.aux_op)
    assert st == g.OK, g.status_string(st)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    Dh = D.cpu()
    return inputs.bits(Dh.t().contiguous() if col_major_cd else Dh)


@pytest.mark.parametrize("op", ["add", "sub", "mul", "div"])
@pytest.mark.parametrize("act", ["relu", "sigmoid"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_aux_tensor_ops(op, act, dtype):
    """D = act(alpha*A.B + beta*C + bias) op Z (EFC epilogue operations)."""
    prob = inputs.random_problem(392, 520, 712, dtype=dtype, alpha=0.5, beta=0.5, act=act,
                                 bias=True, aux_op=op)
    assert_matches_oracle(prob, _run_aux(_plan(prob), prob))


@pytest.mark.parametrize("sched", [g.SCHED_DP, g.SCHED_SK, g.SCHED_SPLIT])
@pytest.mark.parametrize("col_major_cd", [False, True])
def test_aux_under_every_schedule_and_output_layout(sched, col_major_cd):
    prob = inputs.random_problem(296, 264, 2048, dtype="bf16", beta=1.0, act="tanh",
                                 aux_op="mul")
    plan = _plan(prob, layout_cd=LAYOUT[col_major_cd], schedule=sched)
    d = _run_aux(plan, prob, col_major_cd=col_major_cd)
    assert plan.last_config()["schedule"] == sched
    assert_matches_oracle(prob, d)


def test_aux_with_ragged_n_and_k_zero():
    prob = inputs.random_problem(75, 136, 200, beta=1.0, act="relu", aux_op="sub")
    assert_matches_oracle(prob, _run_aux(_plan(prob), prob))
    # N = 136 ends inside the last 64-column chunk; K = 0 runs the reduction kernel alone
    prob0 = inputs.random_problem(40, 72, 0, beta=0.75, act="sigmoid", aux_op="div")
    prob0.A = torch.empty(40, 0, dtype=torch.float16)
    prob0.B = torch.empty(0, 72, dtype=torch.float16)
    assert_matches_oracle(prob0, _run_aux(_plan(prob0), prob0))


def test_aux_argument_errors():
    prob = inputs.random_problem(64, 128, 64, aux_op="add")
    plan = _plan(prob)
    A, B = prob.A.cuda(), prob.B.cuda()
    D = torch.empty(64, 128, dtype=torch.float16, device="cuda")
    Z = prob.aux.cuda()
    run = lambda **kw: g.gemm_run_args(plan.handle, A, B, None, D, 64, 128, 64, 1.0, 0.0, **kw)
    assert run(aux=None, aux_op="add") == g.ERR_INVALID_ARG
    assert run(aux=Z, aux_op=7) == g.ERR_INVALID_ARG
    assert run(aux=Z, aux_op="add", ldaux=100) == g.ERR_INVALID_ARG   # < N
    assert run(aux=Z, aux_op="add", ldaux=132) == g.ERR_ALIGNMENT     # 264 bytes
    assert run(aux=Z, aux_op="add") == g.OK


@pytest.mark.parametrize("act", ["sigmoid", "tanh"])
@pytest.mark.parametrize("sched", [g.SCHED_DP, g.SCHED_SK, g.SCHED_SPLIT])
def test_pre_activation_output_matches_oracle(act, sched):
    """Random operands: Y (pre-activation) against the oracle's linear
    epilogue, D against the full one, with C, a bias and Z."""
    import copy
    prob = inputs.random_problem(392, 520, 1096, dtype="f16", alpha=0.75, beta=0.5, act=act,
                                 bias=True, aux_op="add")
    plan = _plan(prob, schedule=sched)
    A, B, C, Z = prob.A.cuda(), prob.B.cuda(), prob.C.cuda(), prob.aux.cuda()
    D = torch.full((prob.M, prob.N), float("nan"), dtype=torch.float16, device="cuda")
    Y = torch.full_like(D, float("nan"))
    st = g.gemm_run_args(plan.handle, A, B, C, D, prob.M, prob.N, prob.K, prob.alpha,
                         prob.beta, bias=prob.bias.cuda(), aux=Z, aux_op="add", pre=Y)
    assert st == g.OK
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    assert_matches_oracle(prob, inputs.bits(D.cpu()))
    lin = copy.copy(prob)
    lin.act, lin.relu, lin.aux, lin.aux_op = "linear", False, None, None
    assert_matches_oracle(lin, inputs.bits(Y.cpu()))


def test_pre_activation_argument_errors():
    prob = inputs.random_problem(64, 128, 64)
    plan = _plan(prob)
    A, B = prob.A.cuda(), prob.B.cuda()
    D = torch.empty(64, 128, dtype=torch.float16, device="cuda")
    Y = torch.empty(64, 136, dtype=torch.float16, device="cuda")
    run = lambda **kw: g.gemm_run_args(plan.handle, A, B, None, D, 64, 128, 64, 1.0, 0.0, **kw)
    assert run(pre=Y, ldpre=100) == g.ERR_INVALID_ARG    # below N
    assert run(pre=Y, ldpre=132) == g.ERR_ALIGNMENT      # 264 bytes
    assert run(pre=Y.view(-1)[4:], ldpre=136) == g.ERR_ALIGNMENT
    assert run(pre=Y, ldpre=136) == g.OK

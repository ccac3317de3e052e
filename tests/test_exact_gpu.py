"""Bit-exact parity on small-integer operands, through every schedule, tile
shape, layout and entry point.

A and B hold integers in [-2, 2] (C, bias and Z small integers too), and alpha,
beta and the fp8 scales are short binary fractions, so every partial sum, every
stream-K / split-K partial and every epilogue step is exact in fp32: whatever
the order of the k terms, the GPU result is one round-to-nearest-even of the
exact value, the same rounding the oracle applies to its exact fp64 sum.  A
dropped, repeated or misplaced k-block, a lost or doubled stream-K partial or a
wrong tile in a grouped table changes many sums by several units and fails the
comparison, which the accuracy bound of the random-input tests cannot promise.

The exact-value cases of the pages are the all-ones examples ("Python
packages associated with CUTLASS", sections "CUTLASS Python Interface" and
"Installation"); these cases extend that check to random integer operands."""
import numpy as np
import pytest
import torch

from dense_gemm_15_gb300 import binding as g
from dense_gemm_15_gb300 import inputs
from helpers import LAYOUT, assert_bit_exact, oracle_bits

pytestmark = pytest.mark.gpu


def _run_args(plan, prob, col_major_cd=False, with_pre=False):
    """Runs `prob` (bias, Z and fp8 scales included) through gemm_run_args;
    returns D as M x N row-major stored bits (and the pre-activation output Y
    the same way with `with_pre`)."""
    A, B = prob.A.cuda(), prob.B.cuda()
    C = prob.C.cuda() if prob.C is not None else None
    Z = prob.aux.cuda() if prob.aux_op else None
    bias = prob.bias.cuda() if prob.bias is not None else None
    dt = inputs.TORCH_DTYPE[prob.d_dtype]
    if col_major_cd:
        C = C.t().contiguous() if C is not None else None
        Z = Z.t().contiguous() if Z is not None else None
        D = torch.full((prob.N, prob.M), float("nan"), dtype=dt, device="cuda")
    else:
        D = torch.full((prob.M, prob.N), float("nan"), dtype=dt, device="cuda")
    Y = torch.full_like(D, float("nan")) if with_pre else None
    sa = sb = None
    if prob.a_dtype == "e4m3":
        sa = torch.tensor([prob.scale_a], dtype=torch.float32, device="cuda")
        sb = torch.tensor([prob.scale_b], dtype=torch.float32, device="cuda")
    st = g.gemm_run_args(plan.handle, A, B, C, D, prob.M, prob.N, prob.K, prob.alpha,
                         prob.beta, scale_a=sa, scale_b=sb, bias=bias, aux=Z,
                         aux_op=prob.aux_op, pre=Y)
    assert st == g.OK, g.status_string(st)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    out = [D.cpu()] + ([Y.cpu()] if with_pre else [])
    out = [inputs.bits(t.t().contiguous() if col_major_cd else t) for t in out]
    return tuple(out) if with_pre else out[0]


def _linear_part(prob):
    """The same problem without activation and auxiliary operation: its D is
    the pre-activation value alpha * s_a * s_b * A.B + beta * C + bias."""
    import copy
    lin = copy.copy(prob)
    lin.act, lin.relu, lin.aux, lin.aux_op = "linear", False, None, None
    return lin


def _plan(prob, layout_cd=g.ROW_MAJOR, **opts):
    plan = g.Plan(prob.a_dtype, prob.d_dtype, epilogue=prob.act,
                  layout_a=LAYOUT[prob.a_col_major], layout_b=LAYOUT[prob.b_col_major],
                  layout_cd=layout_cd)
    for k, v in opts.items():
        plan.set(getattr(g, "OPT_" + k.upper()), v)
    return plan


# ------------------------------------------------------------------ schedules x tiles

TILES = [(1, 128), (1, 256), (2, 256), (2, 128)]


@pytest.mark.parametrize("sched", [g.SCHED_DP, g.SCHED_SK, g.SCHED_SPLIT])
@pytest.mark.parametrize("cg,tile_n", TILES)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_every_schedule_and_tile_bit_exact(sched, cg, tile_n, dtype):
    """520 x 392 x 4160: ragged M and N, 65 k-blocks; stream-K cuts every
    tile over about fifteen units, split-K over several splits."""
    prob = inputs.integer_problem(520, 392, 4160, dtype=dtype, bias=True)
    plan = _plan(prob, schedule=sched, cta_group=cg, tile_n=tile_n)
    d = _run_args(plan, prob)
    cfg = plan.last_config()
    assert (cfg["schedule"], cfg["cta_group"], cfg["tile_n"]) == (sched, cg, tile_n)
    assert_bit_exact(prob, d)


@pytest.mark.parametrize("a_col,b_col", [(True, False), (False, True), (True, True)])
@pytest.mark.parametrize("sched,cg", [(g.SCHED_DP, 2), (g.SCHED_SK, 1), (g.SCHED_SK, 2),
                                      (g.SCHED_SPLIT, 1)])
def test_operand_layouts_bit_exact(a_col, b_col, sched, cg):
    prob = inputs.integer_problem(392, 520, 2112, dtype="bf16", a_col_major=a_col,
                                  b_col_major=b_col)
    plan = _plan(prob, schedule=sched, cta_group=cg)
    assert_bit_exact(prob, _run_args(plan, prob))


@pytest.mark.parametrize("M,N,K,act", [(16, 8192, 2048, "linear"), (300, 1040, 4096, "relu"),
                                       (128, 768, 16384, "linear")])
def test_balanced_split_k_bit_exact(M, N, K, act):
    prob = inputs.integer_problem(M, N, K, dtype="bf16", act=act, bias=True)
    plan = _plan(prob, schedule=g.SCHED_SPLIT, splits=-1)
    d = _run_args(plan, prob)
    assert plan.last_config()["splits"] == 0
    assert_bit_exact(prob, d)


@pytest.mark.parametrize("splits", [2, 7, 33])
def test_split_k_split_counts_bit_exact(splits):
    prob = inputs.integer_problem(256, 264, 8192, dtype="f16")
    plan = _plan(prob, schedule=g.SCHED_SPLIT, splits=splits, cta_group=1)
    d = _run_args(plan, prob)
    assert plan.last_config()["splits"] == splits
    assert_bit_exact(prob, d)


@pytest.mark.parametrize("inline", [1, 2])
@pytest.mark.parametrize("cg,tile_n,swap", [(1, 128, 1), (1, 256, 1), (2, 256, 1), (2, 128, 1),
                                            (1, 0, 2)])
def test_split_k_in_kernel_and_kernel_reduction_bit_exact(inline, cg, tile_n, swap):
    """Split-K reduced by the split that finishes a tile last (inline = 2, one
    launch) or by the reduction kernel (inline = 1, two launches), with C, a
    bias, Z and the pre-activation output."""
    prob = inputs.integer_problem(520, 392, 4160, dtype="bf16", bias=True, aux_op="mul")
    plan = _plan(prob, schedule=g.SCHED_SPLIT, splits=3, cta_group=cg, tile_n=tile_n,
                 swap_ab=swap, splitk_inline=inline)
    d, y = _run_args(plan, prob, with_pre=True)
    cfg = plan.last_config()
    assert cfg["splits"] == 3 and cfg["launches"] == (1 if inline == 2 else 2)
    assert_bit_exact(prob, d)
    assert_bit_exact(_linear_part(prob), y)


def test_split_k_in_kernel_reduction_is_deterministic():
    prob = inputs.random_problem(264, 1032, 8192, dtype="f16", beta=0.5, relu=True)
    plan = _plan(prob, schedule=g.SCHED_SPLIT, splits=4, splitk_inline=2, tile_n=128)
    d1 = _run_args(plan, prob)
    d2 = _run_args(plan, prob)
    assert plan.last_config()["launches"] == 1
    assert np.array_equal(d1, d2)


# ------------------------------------------------------------------ stream-K partitions

@pytest.mark.parametrize("cg,grid", [(1, 4), (2, 8)])
def test_stream_k_tail_head_whole_partition_bit_exact(cg, grid):
    """Four units over six tiles: each unit holds a whole tile and a tail or
    a head piece of a split tile."""
    m = 128 * cg
    prob = inputs.integer_problem(2 * m, 768, 4096, dtype="f16")
    plan = _plan(prob, schedule=g.SCHED_SK, cta_group=cg, grid=grid, tile_n=256)
    d = _run_args(plan, prob)
    assert plan.last_config()["tiles"] == 6
    assert_bit_exact(prob, d)


@pytest.mark.parametrize("cg", [1, 2])
def test_stream_k_owner_finishing_last_bit_exact(cg):
    """Three tiles over five units: the owners hold no head piece, and two
    units publish two partial tiles each."""
    prob = inputs.integer_problem(128 * cg, 768, 4096, dtype="bf16", alpha=-1.25, act="linear")
    plan = _plan(prob, schedule=g.SCHED_SK, cta_group=cg, grid=5 * cg, tile_n=256)
    d1 = _run_args(plan, prob)
    assert_bit_exact(prob, d1)


@pytest.mark.parametrize("cg,units,N", [(1, 4, 200), (2, 4, 200), (1, 3, 392), (2, 3, 392)])
def test_stream_k_owner_that_ends_its_unit_bit_exact(cg, units, N):
    """Owner pieces at the end of their unit add the peers' partials staged in
    the idle TMEM accumulator."""
    prob = inputs.integer_problem(128 * cg - 8, N, 4096, dtype="f16")
    plan = _plan(prob, schedule=g.SCHED_SK, cta_group=cg, grid=units * cg, tile_n=256)
    assert_bit_exact(prob, _run_args(plan, prob))


@pytest.mark.parametrize("waves", [0, 1])
def test_stream_k_after_data_parallel_waves_bit_exact(waves):
    """Tiles beyond the data-parallel waves go to stream-K: 9 x 17 SM-pair
    tiles (about two waves), with and without one data-parallel wave first."""
    prob = inputs.integer_problem(2304, 4352, 1024, dtype="bf16", bias=True)
    plan = _plan(prob, schedule=g.SCHED_SK, sk_dp_waves=waves, cta_group=2)
    assert_bit_exact(prob, _run_args(plan, prob))


# ------------------------------------------------------------------ fp8

@pytest.mark.parametrize("sched", [g.SCHED_DP, g.SCHED_SK, g.SCHED_SPLIT])
@pytest.mark.parametrize("cg", [1, 2])
def test_e4m3_power_of_two_scales_bit_exact(sched, cg):
    """e4m3 integer operands, scales 1/2 and 1/4 (alpha * s_a * s_b = 3/16)."""
    prob = inputs.integer_problem(520, 528, 4224, dtype="e4m3", beta=0.0, scale_a=0.5,
                                  scale_b=0.25, bias=True)
    plan = _plan(prob, schedule=sched, cta_group=cg, tile_n=256)
    assert_bit_exact(prob, _run_args(plan, prob))


# ------------------------------------------------------------------ C / D layout, epilogue

@pytest.mark.parametrize("sched", [g.SCHED_DP, g.SCHED_SK, g.SCHED_SPLIT])
def test_column_major_c_d_bit_exact(sched):
    prob = inputs.integer_problem(392, 264, 4096, dtype="f16", bias=True, aux_op="add")
    plan = _plan(prob, layout_cd=g.COL_MAJOR, schedule=sched)
    assert_bit_exact(prob, _run_args(plan, prob, col_major_cd=True))


@pytest.mark.parametrize("op", ["add", "sub", "mul", "div"])
@pytest.mark.parametrize("sched", [g.SCHED_DP, g.SCHED_SK, g.SCHED_SPLIT])
def test_aux_ops_bit_exact(op, sched):
    prob = inputs.integer_problem(296, 392, 2048, dtype="bf16", bias=True, aux_op=op)
    plan = _plan(prob, schedule=sched)
    assert_bit_exact(prob, _run_args(plan, prob))


def test_k_zero_bit_exact():
    prob = inputs.integer_problem(70, 136, 0, dtype="f16", bias=True, aux_op="mul")
    prob.A = torch.empty(70, 0, dtype=torch.float16)
    prob.B = torch.empty(0, 136, dtype=torch.float16)
    assert_bit_exact(prob, _run_args(_plan(prob), prob))


# ------------------------------------------------------------------ swap-AB (skinny M)

@pytest.mark.parametrize("sched", [g.SCHED_DP, g.SCHED_SK, g.SCHED_SPLIT])
@pytest.mark.parametrize("M", [1, 16, 64, 65, 128])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_swap_ab_bit_exact(sched, M, dtype):
    """D^T = B^T . A^T on 128 x 64 (M <= 64) or 128 x 128 tiles, stored
    transposed: ragged N (1160 = 9 tiles and a bit) and M, with C, a bias and
    an auxiliary tensor read transposed."""
    prob = inputs.integer_problem(M, 1160, 2112, dtype=dtype, bias=True, aux_op="add")
    plan = _plan(prob, schedule=sched, swap_ab=2)
    d = _run_args(plan, prob)
    cfg = plan.last_config()
    assert cfg["swap_ab"] == 1 and cfg["schedule"] == sched
    assert cfg["tile_n"] == (64 if M <= 64 else 128) and cfg["cta_group"] == 1
    assert_bit_exact(prob, d)


@pytest.mark.parametrize("sched", [g.SCHED_DP, g.SCHED_SK, g.SCHED_SPLIT])
@pytest.mark.parametrize("M", [72, 128])
def test_swap_ab_sm_pair_tiles_bit_exact(sched, M):
    """Swap-AB on SM-pair 256 x 128 tiles (each CTA stages 64 of the tokens),
    stored transposed, with C, a bias, Z and the pre-activation output."""
    prob = inputs.integer_problem(M, 1160, 2112, dtype="bf16", bias=True, aux_op="add")
    plan = _plan(prob, schedule=sched, swap_ab=2, cta_group=2)
    d, y = _run_args(plan, prob, with_pre=True)
    cfg = plan.last_config()
    assert cfg["swap_ab"] == 1 and cfg["cta_group"] == 2 and cfg["tile_n"] == 128
    assert_bit_exact(prob, d)
    assert_bit_exact(_linear_part(prob), y)


@pytest.mark.parametrize("a_col,b_col", [(True, False), (False, True), (True, True)])
@pytest.mark.parametrize("sched", [g.SCHED_SK, g.SCHED_SPLIT])
def test_swap_ab_operand_layouts_bit_exact(a_col, b_col, sched):
    prob = inputs.integer_problem(40, 1032, 4096, dtype="bf16", a_col_major=a_col,
                                  b_col_major=b_col, aux_op="mul")
    plan = _plan(prob, schedule=sched, swap_ab=2)
    assert_bit_exact(prob, _run_args(plan, prob))
    assert plan.last_config()["swap_ab"] == 1


@pytest.mark.parametrize("sched", [g.SCHED_DP, g.SCHED_SK, g.SCHED_SPLIT])
def test_swap_ab_column_major_c_d_bit_exact(sched):
    """Column-major C/D already computes D^T; swap-AB then computes D itself
    and stores it transposed into the column-major storage."""
    prob = inputs.integer_problem(24, 1040, 2048, dtype="f16", bias=True, aux_op="sub")
    plan = _plan(prob, layout_cd=g.COL_MAJOR, schedule=sched, swap_ab=2)
    assert_bit_exact(prob, _run_args(plan, prob, col_major_cd=True))
    assert plan.last_config()["swap_ab"] == 0  # two transposes


@pytest.mark.parametrize("M", [16, 128])
@pytest.mark.parametrize("sched", [g.SCHED_SK, g.SCHED_SPLIT])
def test_swap_ab_e4m3_bit_exact(M, sched):
    prob = inputs.integer_problem(M, 1056, 4224, dtype="e4m3", beta=0.0, scale_a=0.5,
                                  scale_b=0.25, bias=True)
    plan = _plan(prob, schedule=sched, swap_ab=2)
    assert_bit_exact(prob, _run_args(plan, prob))
    cfg = plan.last_config()
    assert cfg["swap_ab"] == 1 and cfg["tile_n"] == 128


@pytest.mark.parametrize("M", [16, 128])
def test_swap_ab_is_the_automatic_choice_for_decode_sizes(M):
    prob = inputs.integer_problem(M, 8192, 8192, dtype="bf16", beta=0.0, act="linear")
    plan = _plan(prob)
    d = _run_args(plan, prob)
    assert plan.last_config()["swap_ab"] == 1
    assert_bit_exact(prob, d)


# ------------------------------------------------------------------ pre-activation output

@pytest.mark.parametrize("sched", [g.SCHED_DP, g.SCHED_SK, g.SCHED_SPLIT])
@pytest.mark.parametrize("cg,tile_n", [(1, 256), (2, 256), (2, 128)])
def test_pre_activation_output_bit_exact(sched, cg, tile_n):
    """The auxiliary tensor store: Y = alpha*A.B + beta*C + bias (before the
    ReLU and the auxiliary operation) next to D = relu(Y) * Z, both exact.
    N = 392 ends inside a 64-column chunk (element-wise tail)."""
    prob = inputs.integer_problem(520, 392, 4160, dtype="bf16", bias=True, aux_op="mul")
    plan = _plan(prob, schedule=sched, cta_group=cg, tile_n=tile_n)
    d, y = _run_args(plan, prob, with_pre=True)
    assert_bit_exact(prob, d)
    assert_bit_exact(_linear_part(prob), y)


@pytest.mark.parametrize("swap,col_major_cd", [(2, False), (2, True), (1, True)])
@pytest.mark.parametrize("sched", [g.SCHED_SK, g.SCHED_SPLIT])
def test_pre_activation_output_transposed_bit_exact(swap, col_major_cd, sched):
    """Y under swap-AB and column-major C/D (transposed stores), including the
    split-K reduction kernel's store."""
    prob = inputs.integer_problem(48, 1048, 2112, dtype="f16", bias=True, aux_op="add")
    plan = _plan(prob, layout_cd=LAYOUT[col_major_cd], schedule=sched, swap_ab=swap)
    d, y = _run_args(plan, prob, col_major_cd=col_major_cd, with_pre=True)
    assert_bit_exact(prob, d)
    assert_bit_exact(_linear_part(prob), y)


def test_pre_activation_output_with_k_zero():
    prob = inputs.integer_problem(70, 136, 0, dtype="bf16", bias=True, aux_op="sub")
    prob.A = torch.empty(70, 0, dtype=torch.bfloat16)
    prob.B = torch.empty(0, 136, dtype=torch.bfloat16)
    d, y = _run_args(_plan(prob), prob, with_pre=True)
    assert_bit_exact(prob, d)
    assert_bit_exact(_linear_part(prob), y)


# ------------------------------------------------------------------ grouped and batched

@pytest.mark.parametrize("cg", [1, 2])
def test_grouped_bit_exact(cg):
    sizes = [(64, 256, 1024), (200, 392, 2112), (1, 16, 64), (385, 512, 576), (520, 1040, 1088),
             (256, 256, 4096)]
    probs = [inputs.integer_problem(M, N, K, dtype="f16", seed=i)
             for i, (M, N, K) in enumerate(sizes)]
    plan = _plan(probs[0], cta_group=cg)
    dev = []
    for p in probs:
        dev.append(dict(M=p.M, N=p.N, K=p.K, A=p.A.cuda(), B=p.B.cuda(), C=p.C.cuda(),
                        D=torch.full((p.M, p.N), float("nan"), dtype=torch.float16,
                                     device="cuda")))
    plan.grouped(dev, alpha=probs[0].alpha, beta=probs[0].beta)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    assert plan.last_config()["cta_group"] == cg
    for p, t in zip(probs, dev):
        assert_bit_exact(p, inputs.bits(t["D"].cpu()))


@pytest.mark.parametrize("cg", [1, 2])
def test_grouped_e4m3_per_group_scales_bit_exact(cg):
    """Grouped fp8: every group has its own per-tensor scales of A_g and B_g
    (one group without any), folded into its alpha in the epilogue."""
    sizes = [(64, 256, 1024), (200, 400, 2176), (385, 512, 640), (520, 1040, 1152), (256, 256, 4096)]
    scales = [(0.5, 0.25), (1.0, 2.0), (None, None), (4.0, 0.125), (0.25, None)]
    probs = [inputs.integer_problem(M, N, K, dtype="e4m3", seed=i,
                                    scale_a=sa if sa is not None else 1.0,
                                    scale_b=sb if sb is not None else 1.0)
             for i, ((M, N, K), (sa, sb)) in enumerate(zip(sizes, scales))]
    plan = _plan(probs[0], cta_group=cg)
    dev = []
    for p, (sa, sb) in zip(probs, scales):
        f = lambda v: torch.tensor([v], dtype=torch.float32, device="cuda") if v is not None else None
        dev.append(dict(M=p.M, N=p.N, K=p.K, A=p.A.cuda(), B=p.B.cuda(), C=p.C.cuda(),
                        D=torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16, device="cuda"),
                        scale_a=f(sa), scale_b=f(sb)))
    plan.grouped(dev, alpha=probs[0].alpha, beta=probs[0].beta)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    assert plan.last_config()["cta_group"] == cg
    for p, t in zip(probs, dev):
        assert_bit_exact(p, inputs.bits(t["D"].cpu()))


@pytest.mark.parametrize("dtype,a_col,b_col", [("f16", False, False), ("bf16", True, False),
                                               ("f16", False, True), ("e4m3", False, False)])
def test_grouped_column_major_c_d_bit_exact(dtype, a_col, b_col):
    """Grouped GEMM on a plan with column-major C and D (each group computed as
    D_g^T = B_g^T . A_g^T): ragged groups, fp8 groups with their own scales."""
    sizes = [(64, 256, 1024), (200, 400, 2176), (8, 16, 128), (392, 512, 640)]  # ld = M: M % 8 == 0
    e4 = dtype == "e4m3"
    probs = [inputs.integer_problem(M, N, K, dtype=dtype, seed=10 + i, a_col_major=a_col,
                                    b_col_major=b_col, beta=0.0 if e4 else 0.5,
                                    scale_a=0.5 if e4 else 1.0, scale_b=2.0 if e4 else 1.0)
             for i, (M, N, K) in enumerate(sizes)]
    plan = _plan(probs[0], layout_cd=g.COL_MAJOR)
    dt = inputs.TORCH_DTYPE[probs[0].d_dtype]
    dev = []
    for p in probs:
        f = lambda v: torch.tensor([v], dtype=torch.float32, device="cuda")
        dev.append(dict(M=p.M, N=p.N, K=p.K, A=p.A.cuda(), B=p.B.cuda(),
                        C=p.C.t().contiguous().cuda() if p.C is not None else None,
                        D=torch.full((p.N, p.M), float("nan"), dtype=dt, device="cuda"),
                        scale_a=f(p.scale_a) if e4 else None, scale_b=f(p.scale_b) if e4 else None))
    plan.grouped(dev, alpha=probs[0].alpha, beta=probs[0].beta)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    for p, t in zip(probs, dev):
        assert_bit_exact(p, inputs.bits(t["D"].cpu().t().contiguous()))


def test_grouped_scales_need_an_fp8_plan():
    prob = inputs.integer_problem(64, 256, 1024, dtype="f16")
    plan = _plan(prob)
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    D = torch.empty(64, 256, dtype=torch.float16, device="cuda")
    st = g.grouped_gemm_run(plan.handle, [dict(M=64, N=256, K=1024, A=prob.A.cuda(), B=prob.B.cuda(),
                                               C=None, D=D, scale_a=one)], alpha=1.0, beta=0.0)
    assert st == g.ERR_INVALID_ARG


# ------------------------------------------------------------------ back-to-back launches

def test_back_to_back_dependent_gemms_bit_exact():
    """A chain of GEMMs on one stream with no synchronisation: each reads the
    previous one's D (every GEMM kernel is a programmatic dependent launch that
    waits for the kernel before it before touching global memory), through
    data-parallel, stream-K and split-K-with-reduction-kernel launches."""
    import oracle
    M, K = 256, 64
    p1 = inputs.integer_problem(M, 512, K, dtype="bf16", alpha=1.0, beta=0.0, act="linear", seed=1)
    d1_want = oracle_bits(p1)  # |D1| <= 256: exact in bf16
    # |D2| <= 256 * 512 = 2^17 and |D3| <= 2^17 * 64 = 2^23: every sum exact in fp32
    B2 = inputs.integers((512, 64), -1, 1, "bf16", 8, 77, 0)
    B3 = inputs.integers((64, 640), -1, 1, "bf16", 8, 78, 0)
    plans = [_plan(p1, schedule=g.SCHED_DP), _plan(p1, schedule=g.SCHED_SK, grid=24),
             _plan(p1, schedule=g.SCHED_SPLIT, splits=4, splitk_inline=1, cta_group=1)]
    for plan2 in plans:
        A1, B1 = p1.A.cuda(), p1.B.cuda()
        D1 = torch.full((M, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        D2 = torch.full((M, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
        D3 = torch.full((M, 640), float("nan"), dtype=torch.bfloat16, device="cuda")
        plans[0].run(A1, B1, None, D1, M, 512, K)
        plan2.run(D1, B2.cuda(), None, D2, M, 64, 512)
        plans[0].run(D2, B3.cuda(), None, D3, M, 640, 64)
        torch.cuda.synchronize()
        assert plans[0].query_error() == g.OK and plan2.query_error() == g.OK
        d1 = inputs.bits(D1.cpu())
        assert np.array_equal(d1, d1_want)
        d2_want = oracle.round_to(oracle.gemm(d1_want, "bf16", inputs.bits(B2), "bf16"), "bf16")
        assert np.array_equal(inputs.bits(D2.cpu()), d2_want)
        d3_want = oracle.round_to(oracle.gemm(d2_want, "bf16", inputs.bits(B3), "bf16"), "bf16")
        assert np.array_equal(inputs.bits(D3.cpu()), d3_want)


@pytest.mark.parametrize("sched,opts", [(g.SCHED_SK, dict(grid=40)),
                                        (g.SCHED_SPLIT, dict(splits=5, splitk_inline=2)),
                                        (g.SCHED_SPLIT, dict(splits=5, splitk_inline=1))])
def test_back_to_back_launches_of_one_plan_bit_exact(sched, opts):
    """Three launches of one plan back to back without synchronisation: the
    plan's workspace, flags and counters serve each in turn, so a launch that
    touched them before the previous one finished would corrupt its partials."""
    probs = [inputs.integer_problem(384, 520, 4096, dtype="f16", seed=s) for s in range(3)]
    plan = _plan(probs[0], schedule=sched, cta_group=1, tile_n=128, **opts)
    outs = []
    for p in probs:
        D = torch.full((p.M, p.N), float("nan"), dtype=torch.float16, device="cuda")
        plan.run(p.A.cuda(), p.B.cuda(), p.C.cuda(), D, p.M, p.N, p.K, alpha=p.alpha, beta=p.beta)
        outs.append(D)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    for p, D in zip(probs, outs):
        assert_bit_exact(p, inputs.bits(D.cpu()))


def test_batched_bit_exact():
    batch, M, N, K = 5, 264, 392, 1040
    probs = [inputs.integer_problem(M, N, K, dtype="bf16", seed=b) for b in range(batch)]
    A = torch.stack([p.A for p in probs]).cuda()
    B = torch.stack([p.B for p in probs]).cuda()
    C = torch.stack([p.C for p in probs]).cuda()
    D = torch.full((batch, M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    plan = _plan(probs[0])
    plan.batched(A, B, C, D, M, N, K, batch, M * K, K * N, M * N, M * N,
                 alpha=probs[0].alpha, beta=probs[0].beta)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    Dh = D.cpu()
    for b, p in enumerate(probs):
        assert_bit_exact(p, inputs.bits(Dh[b].contiguous()))


# ------------------------------------------------------------------ special values

def test_relu_of_nan_from_c_stays_nan():
    """ReLU with beta != 0 and NaN entries in C: those elements of D are NaN
    (NaN propagates through ReLU), every other element is bit-exact."""
    prob = inputs.integer_problem(264, 392, 1024, dtype="f16", act="relu")
    C = prob.C.clone()
    nan_at = [(0, 0), (17, 255), (130, 3), (263, 391), (200, 256)]
    for i, j in nan_at:
        C[i, j] = float("nan")
    prob.C = C
    for sched in (g.SCHED_DP, g.SCHED_SK, g.SCHED_SPLIT):
        d = _run_args(_plan(prob, schedule=sched), prob)
        want = oracle_bits(prob)
        isnan = np.isnan(d.view(np.float16))
        assert set(map(tuple, np.argwhere(isnan))) == set(nan_at)
        assert np.array_equal(d[~isnan], want[~isnan])


@pytest.mark.parametrize("sched", [g.SCHED_DP, g.SCHED_SPLIT])
def test_fp16_overflow_rounds_to_inf(sched):
    """Exact sums around the top of fp16: 65504 stays, 65519 rounds down to
    65504, 65520 (half way to 65536) rounds to even, which is infinity, and
    larger sums give +-inf; compared bit for bit with the oracle's rounding."""
    M, N, K = 128, 128, 64
    targets = [65504, 65519, 65520, 65535, 70000, 131072, -65519, -65520, -1000000]
    A = torch.zeros(M, K, dtype=torch.float16)
    B = torch.ones(K, N, dtype=torch.float16)
    # row i of A . B = targets[i]: A[i, :] holds the target as a sum of
    # exactly representable fp16 parts (each rounded toward zero)
    for i, t in enumerate(targets):
        r, k = float(t), 0
        while r != 0.0:
            p = float(np.float16(r))
            if abs(p) > abs(r) or not np.isfinite(p):
                p = float(np.nextafter(np.float16(p if np.isfinite(p) else np.sign(r) * 65504),
                                       np.float16(0)))
            p = max(-65504.0, min(65504.0, p))
            A[i, k] = p
            r -= p
            k += 1
        assert float(A[i].double().sum()) == t
    prob = inputs.Problem("overflow", A, B, None, M, N, K, act="linear")
    d = _run_args(_plan(prob, schedule=sched), prob)
    want = oracle_bits(prob)
    assert np.array_equal(d, want)
    v = d.view(np.float16).astype(np.float64)
    assert np.isposinf(v[2]).all() and np.isposinf(v[5]).all() and np.isneginf(v[7]).all()
    assert (v[1] == 65504).all()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("act", ["sigmoid", "tanh"])
def test_activation_saturation(dtype, act):
    """Pre-activation values of magnitude 20 to 60000: sigmoid gives 0 or 1 and
    tanh +-1 up to the output rounding, never NaN (compared with the oracle's
    value rounded to the output type, allowing one unit of the format in the
    last place for the approximate exponential and tanh)."""
    M, N, K = 128, 64, 16
    vals = [20.0, -20.0, 30.0, -30.0, 88.0, -88.0, 100.0, -100.0, 1000.0, -1000.0, 60000.0,
            -60000.0]
    A = torch.zeros(M, K, dtype=inputs.TORCH_DTYPE[dtype])
    for i, v in enumerate(vals):
        A[i, 0] = v
    B = torch.zeros(K, N, dtype=inputs.TORCH_DTYPE[dtype])
    B[0, :] = 1.0
    prob = inputs.Problem("saturation", A, B, None, M, N, K, act=act, a_dtype=dtype,
                          b_dtype=dtype, c_dtype=dtype, d_dtype=dtype)
    d = _run_args(_plan(prob), prob)
    want = oracle_bits(prob)
    got = torch.from_numpy(d.view(np.int16)).view(inputs.TORCH_DTYPE[dtype]).double().numpy()
    ref = torch.from_numpy(want.view(np.int16)).view(inputs.TORCH_DTYPE[dtype]).double().numpy()
    assert np.isfinite(got).all()
    ulp = 2.0 ** -10 if dtype == "f16" else 2.0 ** -7
    assert np.all(np.abs(got - ref) <= ulp * np.maximum(np.abs(ref), 2.0 ** -14) + 1e-30)
    for i, v in enumerate(vals):
        if act == "sigmoid" and v > 0:
            assert np.all(got[i] == 1.0)
        elif act == "sigmoid":
            # 1 / (1 + e^-v) for v <= -20 is below 2.1e-9: zero in fp16, a tiny
            # (possibly flushed) value in bf16
            assert np.all((got[i] >= 0.0) & (got[i] <= 2.1e-9))
        else:
            assert np.all(got[i] == (1.0 if v > 0 else -1.0))


# ------------------------------------------------------------------ host-buffer entry point

def _run_host(plan, prob, stream=None):
    hA, hB = prob.A.pin_memory(), prob.B.pin_memory()
    hC = prob.C.pin_memory() if prob.C is not None else None
    hD = torch.full((prob.M, prob.N), float("nan"), dtype=inputs.TORCH_DTYPE[prob.d_dtype]).pin_memory()
    st = g.gemm_run_host(plan.handle, hA, hB, hC, hD, prob.M, prob.N, prob.K, prob.alpha,
                         prob.beta, prob.scale_a, prob.scale_b, stream)
    return st, inputs.bits(hD)


@pytest.mark.parametrize("dtype,beta", [("f16", 0.5), ("bf16", 0.0), ("e4m3", 0.0)])
def test_gemm_run_host_bit_exact(dtype, beta):
    """gemm_run_host (host buffers, copies inside the call) against the
    oracle; fp8 with HOST scales 1/2 and 1/4."""
    kw = dict(scale_a=0.5, scale_b=0.25) if dtype == "e4m3" else {}
    prob = inputs.integer_problem(520, 528, 4224, dtype=dtype, beta=beta, act="relu", **kw)
    plan = _plan(prob)
    for _ in range(2):  # the second call reuses the plan's device buffers
        st, d = _run_host(plan, prob)
        assert st == g.OK, g.status_string(st)
        assert_bit_exact(prob, d)


@pytest.mark.parametrize("dtype,M,N", [("bf16", 512, 8192), ("f16", 136, 10000)])
def test_gemm_run_host_column_pipeline_bit_exact(dtype, M, N):
    """Large enough for the column-chunked pipeline (B and D over 64 MiB: 4
    chunks; N = 10000 leaves a ragged last chunk), with C: bit-exact, twice."""
    prob = inputs.integer_problem(M, N, 4096, dtype=dtype, beta=0.5, act="relu")
    plan = _plan(prob)
    want = oracle_bits(prob)
    for _ in range(2):
        st, d = _run_host(plan, prob)
        assert st == g.OK, g.status_string(st)
        assert_bit_exact(prob, d, want=want)


def test_gemm_run_host_k_zero_and_empty():
    prob = inputs.integer_problem(70, 136, 0, dtype="f16", act="relu")
    prob.A = torch.empty(70, 0, dtype=torch.float16)
    prob.B = torch.empty(0, 136, dtype=torch.float16)
    plan = _plan(prob)
    st, d = _run_host(plan, prob)
    assert st == g.OK
    assert_bit_exact(prob, d)
    hD = torch.full((4, 8), 3.0, dtype=torch.float16)
    assert g.gemm_run_host(plan.handle, None, None, None, hD, 0, 8, 16, 1.0, 0.0) == g.OK
    assert torch.all(hD == 3.0)


def test_gemm_run_host_reports_and_clears_a_timeout():
    """A stream-K peer that skips its flag (test hook): gemm_run_host returns
    the device timeout and clears the status word, so the next call is OK."""
    prob = inputs.integer_problem(256, 512, 8192, dtype="f16")
    plan = _plan(prob, schedule=g.SCHED_SK, timeout_us=20000, fault_skip_flag=1)
    st, _ = _run_host(plan, prob)
    assert st == g.ERR_TIMEOUT
    plan.set(g.OPT_FAULT_SKIP_FLAG, -1)
    st, d = _run_host(plan, prob)
    assert st == g.OK, g.status_string(st)
    assert plan.query_error() == g.OK
    assert_bit_exact(prob, d)

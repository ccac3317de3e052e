"""Parity of the GEMM variants against the oracle: stream-K and split-K
schedules, grouped GEMM, fp8 e4m3 with per-tensor scales, column-major C/D,
padded leading dimensions, K == 0 and the bounded-wait timeout path."""
import re

import numpy as np
import pytest
import torch

from dense_gemm_15_gb300 import binding as g
from dense_gemm_15_gb300 import inputs
from oracle import check
from helpers import (assert_matches_oracle, assert_windows_match_oracle, band_windows, plan_for,
                     run_gpu)

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ schedules

@pytest.mark.parametrize("sched", [g.SCHED_DP, g.SCHED_SK, g.SCHED_SPLIT])
@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("shape", [(256, 256, 4096), (640, 520, 1000), (130, 1032, 2056)])
def test_schedules_match_oracle(sched, tile_n, shape):
    M, N, K = shape
    prob = inputs.random_problem(M, N, K, beta=0.5, alpha=1.5, relu=True)
    plan = plan_for(prob, schedule=sched, tile_n=tile_n)
    d = run_gpu(plan, prob)
    cfg = plan.last_config()
    assert cfg["schedule"] == sched
    assert_matches_oracle(prob, d)


def test_stream_k_is_deterministic_and_agrees_with_data_parallel():
    prob = inputs.random_problem(384, 768, 8192, beta=1.0)
    sk = plan_for(prob, schedule=g.SCHED_SK)
    d1 = run_gpu(sk, prob)
    d2 = run_gpu(sk, prob)
    assert np.array_equal(d1, d2)
    dp = run_gpu(plan_for(prob, schedule=g.SCHED_DP), prob)
    assert_matches_oracle(prob, d1)
    assert_matches_oracle(prob, dp)


def test_split_k_is_deterministic():
    prob = inputs.random_problem(256, 256, 16384, beta=1.0)
    plan = plan_for(prob, schedule=g.SCHED_SPLIT, splits=12)
    d1 = run_gpu(plan, prob)
    d2 = run_gpu(plan, prob)
    assert plan.last_config()["splits"] == 12
    assert np.array_equal(d1, d2)
    assert_matches_oracle(prob, d1)


@pytest.mark.parametrize("shape", [(256, 256, 65536), (1536, 1536, 16384), (3000, 5000, 7000)])
def test_streamk_stress_configs(shape):
    prob = inputs.config5a(*shape)
    d = run_gpu(plan_for(prob), prob)
    assert_windows_match_oracle(prob, d, band_windows(prob.M, band=256, span=8))


# ------------------------------------------------------------------ layouts and edges

def test_column_major_c_and_d():
    prob = inputs.random_problem(200, 136, 96, beta=0.5, alpha=-1.0)
    plan = g.Plan("f16", layout_cd=g.COL_MAJOR)
    A, B = prob.A.cuda(), prob.B.cuda()
    Ct = prob.C.t().contiguous().cuda()          # column-major storage of C
    Dt = torch.empty(prob.N, prob.M, dtype=torch.float16, device="cuda")
    plan.run(A, B, Ct, Dt, prob.M, prob.N, prob.K, alpha=prob.alpha, beta=prob.beta)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    assert_matches_oracle(prob, inputs.bits(Dt.t().contiguous().cpu()))


def test_padded_leading_dimensions():
    M, N, K = 97, 131, 77
    prob = inputs.random_problem(M, N, K, beta=1.0)
    lda, ldb, ldd = 88, 136, 144  # elements; 16-byte multiples
    A = torch.zeros(M, lda, dtype=torch.float16)
    A[:, :K] = prob.A
    B = torch.zeros(K, ldb, dtype=torch.float16)
    B[:, :N] = prob.B
    C = torch.zeros(M, ldd, dtype=torch.float16)
    C[:, :N] = prob.C
    D = torch.full((M, ldd), 7.0, dtype=torch.float16, device="cuda")
    plan = g.Plan("f16")
    plan.run(A.cuda(), B.cuda(), C.cuda(), D, M, N, K, alpha=1.0, beta=1.0, lda=lda, ldb=ldb,
             ldc=ldd, ldd=ldd)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    Dc = D.cpu()
    assert torch.all(Dc[:, N:] == 7.0), "padding columns of D were written"
    assert_matches_oracle(prob, inputs.bits(Dc[:, :N].contiguous()))


def test_k_zero_gives_beta_c():
    M, N = 70, 136
    C = inputs.uniform((M, N), -2, 2, "f16", 91, 1)
    plan = g.Plan("f16", relu=True)
    D = torch.empty(M, N, dtype=torch.float16, device="cuda")
    dummy = torch.empty(8, dtype=torch.float16, device="cuda")
    plan.run(dummy, dummy, C.cuda(), D, M, N, 0, alpha=3.0, beta=0.5)
    torch.cuda.synchronize()
    want = torch.relu(C.to(torch.float64) * 0.5).to(torch.float16)
    assert np.array_equal(inputs.bits(D.cpu()), inputs.bits(want))


def test_empty_problem_is_a_no_op():
    plan = g.Plan("f16")
    D = torch.full((4, 8), 3.0, dtype=torch.float16, device="cuda")
    st = g.gemm_run(plan.handle, None, None, None, D, 0, 8, 16, 1.0, 0.0)
    assert st == g.OK
    st = g.gemm_run(plan.handle, None, None, None, D, 4, 0, 16, 1.0, 0.0)
    assert st == g.OK
    torch.cuda.synchronize()
    assert torch.all(D == 3.0)


def test_argument_errors_launch_nothing():
    plan = g.Plan("f16")
    a = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    d = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    h = plan.handle
    assert g.gemm_run(h, a, a, None, d, -1, 64, 64, 1.0, 0.0) == g.ERR_INVALID_ARG
    assert g.gemm_run(h, a, a, None, None, 64, 64, 64, 1.0, 0.0) == g.ERR_INVALID_ARG
    assert g.gemm_run(h, a, a, None, d, 64, 64, 64, 1.0, 1.0) == g.ERR_INVALID_ARG  # C missing
    odd = a.view(-1)[1:].data_ptr()  # 2-byte offset: not 16-byte aligned
    assert g.gemm_run(h, odd, a, None, d, 8, 8, 8, 1.0, 0.0) == g.ERR_ALIGNMENT
    assert g.gemm_run_ex(h, a, 63, a, 64, None, 64, d, 64, 8, 8, 63, 1.0, 0.0) == g.ERR_ALIGNMENT
    assert g.gemm_run_ex(h, a, 8, a, 64, None, 64, d, 64, 8, 8, 16, 1.0, 0.0) == g.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(d == 0)


# ------------------------------------------------------------------ grouped

def _run_grouped(probs, plan):
    dev = []
    for p in probs:
        A, B = p.A.cuda(), p.B.cuda()
        C = p.C.cuda() if p.C is not None else None
        D = torch.empty(p.M, p.N, dtype=inputs.TORCH_DTYPE[p.d_dtype], device="cuda")
        dev.append(dict(M=p.M, N=p.N, K=p.K, A=A, B=B, C=C, D=D))
    plan.grouped(dev, alpha=probs[0].alpha, beta=probs[0].beta)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    return [inputs.bits(t["D"].cpu()) for t in dev]


def test_grouped_small_groups_match_oracle():
    sizes = [(64, 256, 128), (200, 136, 264), (1, 8, 8), (385, 512, 72), (128, 1032, 520)]
    probs = []
    for i, (M, N, K) in enumerate(sizes):
        p = inputs.random_problem(M, N, K, beta=0.5, alpha=1.5, relu=True, seed=i)
        probs.append(p)
    plan = g.Plan("f16", relu=True)
    outs = _run_grouped(probs, plan)
    for p, d in zip(probs, outs):
        assert_matches_oracle(p, d)


def test_grouped_equals_per_group_dense_bitwise():
    probs = inputs.config4(groups=6, N=512, K=256, m_sizes=[64, 300, 129, 1000, 7, 512])
    plan = g.Plan("f16")
    plan.set(g.OPT_SCHEDULE, g.SCHED_DP)
    grouped = _run_grouped(probs, plan)
    for p, d in zip(probs, grouped):
        assert np.array_equal(d, run_gpu(plan, p))


def test_grouped_config4_full():
    probs = inputs.config4()
    plan = g.Plan("f16")
    outs = _run_grouped(probs, plan)
    cfg = plan.last_config()
    rows = 128 * cfg["cta_group"]
    assert cfg["tiles"] == sum(((p.M + rows - 1) // rows) * 16 for p in probs)
    for i, p in enumerate(probs):  # every group, one window in each 256-row band
        assert_windows_match_oracle(p, outs[i], band_windows(p.M, band=256, span=4, seed=i))


@pytest.mark.parametrize("dtype,a_col,b_col", [("f16", False, False), ("bf16", True, False),
                                               ("f16", False, True), ("e4m3", False, False)])
def test_grouped_on_sm_pair_tiles(dtype, a_col, b_col):
    """Groups of ragged M (down to 1 row) on 256 x 256 SM-pair tiles.  N and K
    are multiples of 16 (fp8 rows), M of 8 where A is column-major."""
    ms = [64, 200, 8, 392, 520] if a_col else [64, 200, 1, 385, 520]
    sizes = list(zip(ms, [256, 272, 16, 512, 1040], [128, 400, 128, 144, 528]))
    probs = [inputs.random_problem(M, N, K, dtype=dtype, beta=0.0 if dtype == "e4m3" else 0.5,
                                   alpha=1.5, relu=True, a_col_major=a_col, b_col_major=b_col,
                                   seed=i) for i, (M, N, K) in enumerate(sizes)]
    plan = plan_for(probs[0], cta_group=2)
    outs = _run_grouped(probs, plan)
    cfg = plan.last_config()
    assert cfg["cta_group"] == 2 and cfg["tile_m"] == 256
    assert cfg["tiles"] == sum(((M + 255) // 256) * ((N + 255) // 256) for M, N, _ in sizes)
    for p, d in zip(probs, outs):
        assert_matches_oracle(p, d)


def test_grouped_skips_empty_groups_and_rejects_k_zero():
    plan = g.Plan("f16")
    a = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    d = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    assert g.grouped_gemm_run(plan.handle, [(0, 64, 64, a, a, None, d)]) == g.OK
    assert g.grouped_gemm_run(plan.handle, [(64, 64, 0, a, a, None, d)]) == g.ERR_UNSUPPORTED
    assert g.grouped_gemm_run(plan.handle, []) == g.OK


# ------------------------------------------------------------------ fp8

@pytest.mark.parametrize("scales", [(1.0, 1.0), (0.5, 0.25), (0.37, 1.7)])
def test_e4m3_scales(scales):
    prob = inputs.random_problem(300, 272, 528, dtype="e4m3", scale_a=scales[0],
                                 scale_b=scales[1])
    assert_matches_oracle(prob, run_gpu(plan_for(prob), prob, scales_dev=True))


@pytest.mark.parametrize("a_col,b_col", [(False, False), (True, False), (False, True), (True, True)])
def test_e4m3_layouts(a_col, b_col):
    prob = inputs.random_problem(256, 384, 256, dtype="e4m3", a_col_major=a_col, b_col_major=b_col)
    assert_matches_oracle(prob, run_gpu(plan_for(prob), prob))


def test_e4m3_8192_sampled_rows():
    prob = inputs.config5b(scale_a=0.37, scale_b=1.7)
    d = run_gpu(plan_for(prob), prob, scales_dev=True)
    assert_windows_match_oracle(prob, d, band_windows(prob.M, band=256, span=8))


# ------------------------------------------------------------------ Llama-70B shapes

@pytest.mark.parametrize("layer", list(inputs.LLAMA70B_LAYERS))
def test_llama70b_layers(layer):
    """Every token count of one layer, the weight generated once."""
    K, N = inputs.LLAMA70B_LAYERS[layer]
    W = None
    plan = None
    for M in inputs.LLAMA70B_TOKENS:
        prob = inputs.config3(M, layer) if W is None else None
        if W is None:
            W = prob.B
        else:
            X = inputs.normal((M, K), 1.0, "bf16", 3, 100000 * list(inputs.LLAMA70B_LAYERS).index(layer) + M)
            prob = inputs.Problem("bf16_llama70b_%s_m%d" % (layer, M), X, W, None, M, N, K,
                                  a_dtype="bf16", b_dtype="bf16", c_dtype="bf16", d_dtype="bf16")
        plan = plan or plan_for(prob)
        d = run_gpu(plan, prob)
        assert plan.last_config()["swap_ab"] == (1 if M <= 128 else 0)
        # one window in every 256-row band (each M-tile band of the kernels)
        assert_windows_match_oracle(prob, d, band_windows(M, band=256, span=4, seed=M))


# ------------------------------------------------------------------ bounded waits

def test_stream_k_peer_that_never_publishes_times_out_and_gpu_stays_usable():
    """A stream-K peer skips its partial-ready flag (test hook): the owner's
    bounded wait runs out, the kernel records a timeout and returns; the next
    GEMM on the same plan is correct."""
    prob = inputs.random_problem(256, 512, 8192, beta=1.0)
    plan = plan_for(prob, schedule=g.SCHED_SK, timeout_us=20000, fault_skip_flag=1)
    A, B, C = prob.A.cuda(), prob.B.cuda(), prob.C.cuda()
    D = torch.empty(prob.M, prob.N, dtype=torch.float16, device="cuda")
    plan.run(A, B, C, D, prob.M, prob.N, prob.K, alpha=1.0, beta=1.0)
    torch.cuda.synchronize()
    assert plan.query_error() == g.ERR_TIMEOUT
    assert plan.query_error() == g.OK  # cleared on read
    plan.set(g.OPT_FAULT_SKIP_FLAG, -1)
    assert_matches_oracle(prob, run_gpu(plan, prob))


@pytest.mark.parametrize("a_col,b_col", [(False, False), (False, True), (True, False)])
def test_nan_padding_never_leaks(a_col, b_col):
    """Operands whose leading dimension exceeds the logical extent, with NaN in
    the padding: no padding element may reach D, and no D element beyond N may
    be written.  K, N and M are not multiples of 8."""
    M, N, K = 75, 131, 77
    prob = inputs.random_problem(M, N, K, beta=1.0, a_col_major=a_col, b_col_major=b_col)
    pad = 96  # rounded-up leading extent (multiple of 8 elements)

    def padded(t, rows, cols):
        out = torch.full((rows, cols), float("nan"), dtype=torch.float16)
        out[:t.shape[0], :t.shape[1]] = t
        return out

    if a_col:
        A = padded(prob.A, K, pad)      # storage K x M (column-major A), ld = pad >= M
        lda = pad
    else:
        A = padded(prob.A, M, pad)      # storage M x K, ld = pad >= K
        lda = pad
    if b_col:
        B = padded(prob.B, N, pad)      # storage N x K (column-major B)
        ldb = pad
    else:
        B = padded(prob.B, K, 136)      # storage K x N
        ldb = 136
    C = padded(prob.C, M, 136)
    D = torch.full((M, 136), 7.0, dtype=torch.float16, device="cuda")
    plan = g.Plan("f16", layout_a=g.COL_MAJOR if a_col else g.ROW_MAJOR,
                  layout_b=g.COL_MAJOR if b_col else g.ROW_MAJOR)
    plan.run(A.cuda(), B.cuda(), C.cuda(), D, M, N, K, alpha=1.0, beta=1.0, lda=lda, ldb=ldb,
             ldc=136, ldd=136)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    Dc = D.cpu()
    assert torch.all(Dc[:, N:] == 7.0), "columns beyond N were written"
    assert torch.isfinite(Dc[:, :N]).all(), "padding leaked into D"
    assert_matches_oracle(prob, inputs.bits(Dc[:, :N].contiguous()))


# ------------------------------------------------------------------ SM-pair tiles

@pytest.mark.parametrize("sched", [g.SCHED_DP, g.SCHED_SK, g.SCHED_SPLIT])
@pytest.mark.parametrize("shape", [(512, 512, 1024), (300, 784, 2064), (1000, 272, 528)])
@pytest.mark.parametrize("dtype", ["f16", "bf16", "e4m3"])
def test_sm_pair_tiles(sched, shape, dtype):
    """256 x 256 tiles computed by an SM pair (tcgen05 cta_group::2)."""
    M, N, K = shape
    prob = inputs.random_problem(M, N, K, dtype=dtype, beta=0.5, alpha=1.5, relu=True)
    plan = plan_for(prob, schedule=sched, cta_group=2)
    d = run_gpu(plan, prob)
    cfg = plan.last_config()
    assert cfg["cta_group"] == 2 and cfg["tile_m"] == 256 and cfg["schedule"] == sched
    assert_matches_oracle(prob, d)


@pytest.mark.parametrize("a_col,b_col", [(True, False), (False, True), (True, True)])
def test_sm_pair_tiles_layouts(a_col, b_col):
    prob = inputs.random_problem(640, 512, 768, beta=1.0, a_col_major=a_col, b_col_major=b_col)
    plan = plan_for(prob, cta_group=2)
    assert_matches_oracle(prob, run_gpu(plan, prob))
    assert plan.last_config()["cta_group"] == 2


def test_sm_pair_tiles_chosen_for_large_problems_and_deterministic():
    prob = inputs.random_problem(4096, 4096, 2048, dtype="bf16")
    plan = plan_for(prob)
    d1 = run_gpu(plan, prob)
    assert plan.last_config()["cta_group"] == 2
    d2 = run_gpu(plan, prob)
    assert np.array_equal(d1, d2)
    assert_windows_match_oracle(prob, d1, band_windows(prob.M, band=256, span=8))


def test_timeline_trace_covers_every_k_block_once():
    prob = inputs.random_problem(512, 768, 4096, beta=1.0)
    plan = plan_for(prob, schedule=g.SCHED_SK, cta_group=2, trace_items=16)
    assert_matches_oracle(prob, run_gpu(plan, prob))
    tr = g.gemm_plan_trace(plan.handle)
    cfg = plan.last_config()
    assert tr.shape == (cfg["grid"], 17, 8)
    kb_total = (4096 + 63) // 64
    covered = {}
    for cta in range(tr.shape[0]):
        hdr = tr[cta, 0]
        assert hdr[0] > 0 and hdr[2] >= hdr[0]
        assert hdr[4] == 1, "the final CTA barrier did not order the epilogue before thread 0"
        if cta % 2:  # the pair's second CTA mirrors the first one's items
            continue
        for rec in tr[cta, 1:]:
            if rec[4] == 0:
                continue
            tile = int(rec[0] & 0xffffffff)
            kb0, kb1 = int(rec[1] & 0xffffffff), int(rec[1] >> 32)
            assert rec[2] <= rec[3] and rec[4] <= rec[6]
            covered.setdefault(tile, []).append((kb0, kb1))
    assert len(covered) == cfg["tiles"]
    for tile, parts in covered.items():
        parts.sort()
        assert parts[0][0] == 0 and parts[-1][1] == kb_total
        assert all(a[1] == b[0] for a, b in zip(parts, parts[1:]))


def _sk_items(tr, cta, k_blocks):
    """(piece positions, kinds) of one CTA's traced items: T a tile's tail
    (k0 > 0), H its head (k0 = 0, ends inside), F whole; P a peer, O the owner."""
    pos, kinds = "", ""
    for rec in tr[cta, 1:]:
        if rec[4] == 0:
            continue
        kb0, kb1 = int(rec[1] & 0xffffffff), int(rec[1] >> 32)
        pos += "T" if kb0 > 0 else ("F" if kb1 == k_blocks else "H")
        kinds += "FPOS"[int(rec[0] >> 32)]
    return pos, kinds


@pytest.mark.parametrize("M,N,K,act", [(16, 8192, 2048, "linear"), (300, 1040, 4096, "relu"),
                                       (128, 768, 16384, "tanh")])
def test_balanced_split_k(M, N, K, act):
    """Balanced split-K (splits = -1) cuts the k iterations of all tiles evenly
    over every SM (32, 15 and 3 tiles; in the last case each tile's pieces come
    from about 50 units) and the reduction kernel finds each tile's pieces from
    the partition."""
    prob = inputs.random_problem(M, N, K, dtype="bf16", beta=0.5, act=act, bias=True)
    plan = plan_for(prob, schedule=g.SCHED_SPLIT, splits=-1)
    A, B, C = prob.A.cuda(), prob.B.cuda(), prob.C.cuda()
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    assert g.gemm_run_args(plan.handle, A, B, C, D, M, N, K, prob.alpha, prob.beta,
                           bias=prob.bias.cuda()) == g.OK
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    cfg = plan.last_config()
    assert cfg["schedule"] == g.SCHED_SPLIT and cfg["splits"] == 0 and cfg["launches"] == 2
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert cfg["grid"] == n_sms
    assert_matches_oracle(prob, inputs.bits(D.cpu()))
    D2 = torch.empty_like(D)
    g.gemm_run_args(plan.handle, A, B, C, D2, M, N, K, prob.alpha, prob.beta,
                    bias=prob.bias.cuda())
    torch.cuda.synchronize()
    assert torch.equal(D, D2), "balanced split-K is not deterministic"


@pytest.mark.parametrize("cg,grid", [(1, 4), (2, 8)])
def test_stream_k_takes_tail_then_head_then_whole_tiles(cg, grid):
    """Four units over six tiles of 64 k-blocks: 96 k-blocks each, so every
    unit holds a whole tile and a tail or a head piece; each unit runs its
    tail piece, then its head piece, then its whole tiles.  Head and tail of a
    split tile finish together here, and the lower unit owns the tile."""
    m = 128 * cg
    prob = inputs.random_problem(2 * m, 768, 4096, beta=1.0, relu=True)
    plan = plan_for(prob, schedule=g.SCHED_SK, cta_group=cg, grid=grid, trace_items=8)
    assert_matches_oracle(prob, run_gpu(plan, prob))
    cfg = plan.last_config()
    assert cfg["grid"] == grid and cfg["tiles"] == 6
    tr = g.gemm_plan_trace(plan.handle)
    items = [_sk_items(tr, cta, 64) for cta in range(0, grid, cg)]
    assert all(re.fullmatch(r"T?H?F*", pos) for pos, _ in items), items
    assert items == [("HF", "OF"), ("TF", "PF"), ("HF", "OF"), ("TF", "PF")]


@pytest.mark.parametrize("cg", [1, 2])
def test_stream_k_owner_is_the_holder_that_finishes_last(cg):
    """Three tiles over five units (ranges 0/38/76/115/153/192 of 64-k-block
    tiles): tile 1 is held by units 1 (head, 12 k-blocks after a 26-k-block
    tail), 2 (39, its only piece) and 3 (13); tile 2 by units 3 (head, 25 after
    13) and 4 (39).  Units 2 and 4 finish last and own tiles 1 and 2 although
    they hold no head piece; units 1 and 3 each publish two partial tiles."""
    prob = inputs.random_problem(128 * cg, 768, 4096, beta=0.5, alpha=-1.25, relu=False)
    plan = plan_for(prob, schedule=g.SCHED_SK, cta_group=cg, grid=5 * cg, tile_n=256,
                    trace_items=4)
    d = run_gpu(plan, prob)
    assert_matches_oracle(prob, d)
    assert np.array_equal(d, run_gpu(plan, prob)), "stream-K fix-up is not deterministic"
    tr = g.gemm_plan_trace(plan.handle)
    items = [_sk_items(tr, u * cg, 64) for u in range(5)]
    assert items == [("H", "O"), ("TH", "PP"), ("T", "O"), ("TH", "PP"), ("T", "O")], items


@pytest.mark.parametrize("cg,units,N", [(1, 4, 200), (2, 4, 200), (1, 3, 392), (2, 3, 392)])
def test_stream_k_owner_that_ends_its_unit(cg, units, N):
    """Owner pieces that are the last item of their unit stage the peers'
    partial sum in the idle TMEM accumulator: one tile over four units (three
    peers) and two tiles over three units (one peer each)."""
    prob = inputs.random_problem(128 * cg - 8, N, 4096, beta=0.5, alpha=1.5, relu=True)
    plan = plan_for(prob, schedule=g.SCHED_SK, cta_group=cg, grid=units * cg, tile_n=256,
                    trace_items=4)
    d = run_gpu(plan, prob)
    assert_matches_oracle(prob, d)
    assert np.array_equal(d, run_gpu(plan, prob)), "stream-K fix-up is not deterministic"
    cfg = plan.last_config()
    assert cfg["grid"] == units * cg and cfg["schedule"] == g.SCHED_SK
    tr = g.gemm_plan_trace(plan.handle)
    kinds = ["".join("FPOS"[int(rec[0] >> 32)] for rec in tr[u * cg, 1:] if rec[4] != 0)
             for u in range(units)]
    assert kinds == (["O", "P", "P", "P"] if units == 4 else ["O", "PO", "P"]), kinds


@pytest.mark.parametrize("sched", [g.SCHED_DP, g.SCHED_SK, g.SCHED_SPLIT])
@pytest.mark.parametrize("dtype,a_col,b_col", [("f16", False, False), ("bf16", True, False),
                                               ("f16", False, True), ("bf16", True, True)])
def test_sm_pair_tiles_256x128(sched, dtype, a_col, b_col):
    """256 x 128 tiles on an SM pair (each CTA stages 64 columns of B)."""
    prob = inputs.random_problem(520, 392, 1096, dtype=dtype, beta=0.5, alpha=1.5, relu=True,
                                 a_col_major=a_col, b_col_major=b_col)
    plan = plan_for(prob, schedule=sched, cta_group=2, tile_n=128)
    d = run_gpu(plan, prob)
    cfg = plan.last_config()
    assert cfg["cta_group"] == 2 and cfg["tile_m"] == 256 and cfg["tile_n"] == 128
    assert_matches_oracle(prob, d)

"""Block-scaled GEMM (MXFP8, MXFP4, NVFP4: the _scaled_mm formats of
"Generating State-of-the-Art GEMMs with TorchInductor's CuteDSL backend",
section 5.1) against the oracle, through the C ABI.

The operands are stored on the host in the layout the entry point takes
(inputs.block_scaled_storage): A row-major and B column-major (both K
contiguous), fp4 codes packed two per byte, scale factors in the 128 x 4
blocked atom layout.  The oracle takes the codes one per byte and the scales
as plain M x K/block and K/block x N arrays."""
import numpy as np
import pytest
import torch

from dense_gemm_15_gb300 import binding as g
from dense_gemm_15_gb300 import inputs
from helpers import assert_bit_exact, assert_matches_oracle

pytestmark = pytest.mark.gpu

def device_operands(prob):
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return tuple(dev(x) for x in inputs.block_scaled_storage(prob))


def run_scaled(prob, epilogue="linear", C=None, bias=None, tile_n=0, cta_group=0):
    kind = g.SCALE_NV if prob.block_scales[2] == "e4m3" else g.SCALE_MX
    plan = g.Plan(prob.a_dtype, "bf16", epilogue=epilogue, layout_a=g.ROW_MAJOR,
                  layout_b=g.COL_MAJOR)
    if tile_n:
        plan.set(g.OPT_TILE_N, tile_n)
    if cta_group:
        plan.set(g.OPT_CTA_GROUP, cta_group)
    A, B, SFA, SFB = device_operands(prob)
    D = torch.full((prob.M, prob.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = g.gemm_run_block_scaled(plan.handle, A, B, SFA, SFB, D, prob.M, prob.N, prob.K,
                                 scale_kind=kind, C=C.cuda() if C is not None else None,
                                 alpha=prob.alpha, beta=prob.beta,
                                 bias=bias.cuda() if bias is not None else None)
    assert st == g.OK, g.status_string(st)
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK
    cfg = plan.last_config()
    assert cfg["tile_n"] == (tile_n or 256) and cfg["launches"] == 1
    # default: SM pairs for MXFP8, one SM for the fp4 kinds
    want_cg = cta_group or (1 if tile_n == 128 or prob.a_dtype == "e2m1" else 2)
    assert cfg["cta_group"] == want_cg and cfg["tile_m"] == 128 * want_cg
    return inputs.bits(D.cpu())


FORMATS = [("e4m3", 32, "ue8m0"), ("e5m2", 32, "ue8m0"), ("e2m1", 32, "ue8m0"),
           ("e2m1", 16, "e4m3")]


# (tile_n, cta_group): one-SM 128 x {128, 256}, SM-pair 256 x {256, 128}
TILES = [(128, 1), (256, 1), (256, 2), (128, 2)]


@pytest.mark.parametrize("tile_n,cta_group", TILES)
@pytest.mark.parametrize("elem,block,scale", FORMATS)
@pytest.mark.parametrize("shape", [(256, 512, 1024), (200, 392, 512), (130, 296, 1536),
                                   (520, 264, 768)])
def test_block_scaled_matches_oracle(elem, block, scale, shape, tile_n, cta_group):
    """N(0,1) values with a per-block spread of 2^U{-8..8}, quantised by the
    format's own rules; ragged M and N (the second 128-row block of B's
    scales is absent for N = 296 in the last tile)."""
    M, N, K = shape
    prob = inputs.block_scaled_problem(M, N, K, elem=elem, block=block, scale=scale,
                                       alpha=0.75 if scale == "e4m3" else 1.0)
    assert_matches_oracle(prob, run_scaled(prob, tile_n=tile_n, cta_group=cta_group))


@pytest.mark.parametrize("act", ["relu", "tanh"])
@pytest.mark.parametrize("elem,block,scale", FORMATS)
def test_block_scaled_epilogue_matches_oracle(elem, block, scale, act):
    """alpha, beta * C, a bias and an activation after the block-scaled product."""
    M, N, K = 264, 520, 512
    prob = inputs.block_scaled_problem(M, N, K, elem=elem, block=block, scale=scale, alpha=0.5)
    prob.beta = 0.5
    prob.C = inputs.uniform((M, N), -4, 4, "bf16", 12, 1)
    prob.bias = inputs.uniform((N,), -2, 2, "bf16", 12, 2)
    prob.act = act
    assert_matches_oracle(prob, run_scaled(prob, epilogue=act, C=prob.C, bias=prob.bias))


def _exact_problem(elem, block, scale, M, N, K, seed=0):
    """Small-integer (fp8) or fp4-grid operands with power-of-two block scales
    2^{-1, 0, 1}: every product is a short binary fraction and every sum fits
    fp32, so the result is one rounding of the exact value."""
    rng = np.random.default_rng([seed, 13, M, N, K])
    kb = K // block
    if elem == "e2m1":
        qa = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
        qb = rng.integers(0, 16, size=(K, N)).astype(np.uint8)
    else:
        dt = inputs.TORCH_DTYPE[elem] if elem == "e4m3" else torch.float8_e5m2
        qa = torch.from_numpy(rng.integers(-2, 3, size=(M, K)).astype(np.float32)).to(dt).view(torch.uint8).numpy()
        qb = torch.from_numpy(rng.integers(-2, 3, size=(K, N)).astype(np.float32)).to(dt).view(torch.uint8).numpy()
    e_a = rng.integers(-1, 2, size=(M, kb))
    e_b = rng.integers(-1, 2, size=(kb, N))
    if scale == "ue8m0":
        sa, sb = (e_a + 127).astype(np.uint8), (e_b + 127).astype(np.uint8)
    else:  # e4m3 codes of 2^e: exponent field e + 7, no mantissa
        sa, sb = ((e_a + 7) << 3).astype(np.uint8), ((e_b + 7) << 3).astype(np.uint8)
    p = inputs.Problem("exact_%s_%d" % (elem, block), torch.from_numpy(qa), torch.from_numpy(qb),
                       None, M, N, K, a_dtype=elem, b_dtype=elem, c_dtype="bf16", d_dtype="bf16")
    p.block_scales = (torch.from_numpy(sa), torch.from_numpy(sb), scale, block)
    return p


@pytest.mark.parametrize("tile_n,cta_group", TILES)
@pytest.mark.parametrize("elem,block,scale", FORMATS)
def test_block_scaled_bit_exact(elem, block, scale, tile_n, cta_group):
    """392 x 520 x 2048 (ragged in M and N, more k-blocks than pipeline
    stages): equal to the oracle's rounded result bit for bit."""
    prob = _exact_problem(elem, block, scale, 392, 520, 2048)
    d = run_scaled(prob, tile_n=tile_n, cta_group=cta_group)
    import oracle
    a, b = inputs.bits(prob.A), inputs.bits(prob.B)
    sa, sb, sc, blk = prob.block_scales
    want = oracle.round_to(oracle.gemm(a, elem, b, elem, scales=(inputs.bits(sa), inputs.bits(sb),
                                                                  sc, blk)), "bf16")
    assert_bit_exact(prob, d, want=want)


def test_block_scaled_argument_errors():
    prob = _exact_problem("e4m3", 32, "ue8m0", 128, 256, 256)
    A, B, SFA, SFB = device_operands(prob)
    D = torch.empty(128, 256, dtype=torch.bfloat16, device="cuda")
    plan = g.Plan("e4m3", "bf16", layout_a=g.ROW_MAJOR, layout_b=g.COL_MAJOR)
    run = lambda **kw: g.gemm_run_block_scaled(plan.handle, kw.pop("A", A), B, SFA, SFB, D,
                                               kw.pop("M", 128), 256, kw.pop("K", 256), **kw)
    assert run(K=192) == g.ERR_UNSUPPORTED                   # not a multiple of 128
    assert run(scale_kind=g.SCALE_NV) == g.ERR_UNSUPPORTED   # NV scales are fp4-only
    assert run(scale_kind=7) == g.ERR_INVALID_ARG
    assert run(A=A.view(-1)[8:]) == g.ERR_ALIGNMENT
    assert run(M=0) == g.OK
    rowb = g.Plan("e4m3", "bf16")                            # B row-major: not TN
    assert g.gemm_run_block_scaled(rowb.handle, A, B, SFA, SFB, D, 128, 256, 256) == g.ERR_UNSUPPORTED
    fp4 = g.Plan("e2m1", "bf16", layout_a=g.ROW_MAJOR, layout_b=g.COL_MAJOR)
    assert g.gemm_run(fp4.handle, A, B, None, D, 128, 256, 256) == g.ERR_UNSUPPORTED
    assert run() == g.OK
    torch.cuda.synchronize()
    assert plan.query_error() == g.OK

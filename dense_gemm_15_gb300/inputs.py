"""Seeded synthetic inputs for the GEMM workloads.

This module holds random draws and storage casts only -- none of the GEMM
arithmetic.  It is the one piece shared by the tests (which feed the same
tensors to the CUDA path and to the CPU oracle) and the benchmark.

Recipe (the same for every workload):
  * generator ``numpy.random.default_rng([seed, workload_id, tensor_id])``
    (PCG64), seed 0 by default;
  * values are drawn in float64, then rounded to the storage type by a torch
    CPU cast (round to nearest even); fp8 values are clamped to +-448 first;
  * tensors are returned as CPU torch tensors in storage layout (row-major
    unless a column-major layout is asked for, in which case the returned
    tensor is the transpose's row-major storage).

Workload ids (the ``workload_id`` seed component):
  1  fp16 1024^3, D = A.B + C               (case a all ones, case b U[-1,1])
  2  fp16 4096^3, alpha 1.5, beta 0.5, ReLU  (A,B ~ N(0, 1/sqrt(K)), C ~ N(0,1))
  3  bf16 Llama-3.3-70B linear layers        (W ~ N(0, 0.02), X ~ N(0, 1), beta 0)
  4  fp16 grouped, 32 groups, N 4096, K 2048 (M_g ~ U{64..4096}, U[-1,1])
  5  fp16 stream-K shapes (U[-1,1]) and e4m3 8192^3 (N(0,1) clamped to +-448)
  8  small-integer operands (exact-arithmetic parity cases)
  11 block-scaled operands (MX / NVFP4 storage of N(0,1) float32 values with a
     per-block spread of 2^U{-8..8}); the quantisation to codes and block
     scales is storage preparation, like the fp8 cast above: the GEMM takes
     the codes and scales as they are.
"""
from __future__ import annotations

import numpy as np
import torch

TORCH_DTYPE = {
    "f16": torch.float16,
    "bf16": torch.bfloat16,
    "f32": torch.float32,
    "e4m3": torch.float8_e4m3fn,
}

E4M3_MAX = 448.0

# Llama-3.3-70B linear layers as (K, N) of the weight [K, N].
LLAMA70B_LAYERS = {
    "qkv": (8192, 10240),
    "o_proj": (8192, 8192),
    "gate_up": (8192, 57344),
    "down": (28672, 8192),
}
LLAMA70B_TOKENS = (16, 128, 1024, 4096, 8192)

STREAMK_SHAPES = ((256, 256, 65536), (1536, 1536, 16384), (3000, 5000, 7000))


def rng(workload_id: int, tensor_id: int, seed: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, workload_id, tensor_id])


def _store(x64: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x64))
    if dtype == "e4m3":
        t = t.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float32)
    return t.to(TORCH_DTYPE[dtype])


def uniform(shape, lo, hi, dtype, workload_id, tensor_id, seed=0) -> torch.Tensor:
    return _store(rng(workload_id, tensor_id, seed).uniform(lo, hi, size=shape), dtype)


def normal(shape, std, dtype, workload_id, tensor_id, seed=0) -> torch.Tensor:
    return _store(rng(workload_id, tensor_id, seed).normal(0.0, std, size=shape), dtype)


def integers(shape, lo, hi, dtype, workload_id, tensor_id, seed=0) -> torch.Tensor:
    """Uniform integers in [lo, hi] (inclusive), stored in ``dtype`` (exact for
    the small ranges used: every integer of magnitude <= 256 is representable
    in fp16 and bf16, and every one of magnitude <= 16 in e4m3)."""
    return _store(rng(workload_id, tensor_id, seed).integers(lo, hi, size=shape, endpoint=True)
                  .astype(np.float64), dtype)


def ones(shape, dtype) -> torch.Tensor:
    return torch.ones(shape, dtype=TORCH_DTYPE[dtype])


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw stored bits of a CPU tensor as a numpy array (uint16 / uint8)."""
    t = t.contiguous()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.element_size() == 1:
        return t.view(torch.uint8).numpy()
    return t.numpy()


class Problem:
    """One GEMM problem instance: operands in storage form plus scalars."""

    def __init__(self, name, A, B, C, M, N, K, alpha=1.0, beta=0.0, relu=False,
                 a_dtype="f16", b_dtype="f16", c_dtype="f16", d_dtype="f16",
                 a_col_major=False, b_col_major=False, scale_a=1.0, scale_b=1.0,
                 act=None, bias=None, aux=None, aux_op=None):
        self.name = name
        self.A, self.B, self.C = A, B, C
        self.M, self.N, self.K = M, N, K
        self.alpha, self.beta, self.relu = alpha, beta, relu
        # epilogue activation name ("linear", "relu", "sigmoid", "tanh") and an
        # optional per-column bias vector (N elements of the output type)
        self.act = act or ("relu" if relu else "linear")
        self.bias = bias
        # optional auxiliary M x N tensor entering the activated value by
        # aux_op ("add", "sub", "mul", "div")
        self.aux, self.aux_op = aux, aux_op
        self.a_dtype, self.b_dtype = a_dtype, b_dtype
        self.c_dtype, self.d_dtype = c_dtype, d_dtype
        self.a_col_major, self.b_col_major = a_col_major, b_col_major
        self.scale_a, self.scale_b = scale_a, scale_b

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    def __repr__(self):
        return "Problem(%s, M=%d, N=%d, K=%d)" % (self.name, self.M, self.N, self.K)


def _mk(shape_a, shape_b, col_a, col_b):
    sa = (shape_a[1], shape_a[0]) if col_a else shape_a
    sb = (shape_b[1], shape_b[0]) if col_b else shape_b
    return sa, sb


def config1(case: str, seed: int = 0) -> Problem:
    """fp16 1024^3, alpha = beta = 1; case 'a' all ones, case 'b' U[-1,1]."""
    n = 1024
    if case == "a":
        A, B, C = ones((n, n), "f16"), ones((n, n), "f16"), ones((n, n), "f16")
    else:
        A = uniform((n, n), -1, 1, "f16", 1, 0, seed)
        B = uniform((n, n), -1, 1, "f16", 1, 1, seed)
        C = uniform((n, n), -1, 1, "f16", 1, 2, seed)
    return Problem("fp16_1024_%s" % ("ones" if case == "a" else "uniform"),
                   A, B, C, n, n, n, alpha=1.0, beta=1.0)


def config2(M=4096, N=4096, K=4096, strong=False, seed=0, tag=None) -> Problem:
    """fp16, alpha 1.5, beta 0.5, ReLU; A, B ~ N(0, sigma) with sigma = 1/sqrt(K)
    (or K^-1/4 for the 'strong' variant), C ~ N(0, 1)."""
    sigma = K ** -0.25 if strong else K ** -0.5
    wid = 2 if (M, N, K) == (4096, 4096, 4096) else 20 + (M * 7 + N * 3 + K) % 1000
    A = normal((M, K), sigma, "f16", wid, 0, seed)
    B = normal((K, N), sigma, "f16", wid, 1, seed)
    C = normal((M, N), 1.0, "f16", wid, 2, seed)
    name = tag or ("fp16_%dx%dx%d_relu%s" % (M, N, K, "_strong" if strong else ""))
    return Problem(name, A, B, C, M, N, K, alpha=1.5, beta=0.5, relu=True)


def config3(M: int, layer: str, seed=0) -> Problem:
    """bf16 Llama-3.3-70B linear layer: X [M, K] ~ N(0,1), W [K, N] ~ N(0, 0.02),
    beta 0, bf16 out."""
    K, N = LLAMA70B_LAYERS[layer]
    lid = list(LLAMA70B_LAYERS).index(layer)
    X = normal((M, K), 1.0, "bf16", 3, 100000 * lid + M, seed)
    W = normal((K, N), 0.02, "bf16", 3, 100000 * lid + 99999, seed)
    return Problem("bf16_llama70b_%s_m%d" % (layer, M), X, W, None, M, N, K,
                   alpha=1.0, beta=0.0, a_dtype="bf16", b_dtype="bf16",
                   c_dtype="bf16", d_dtype="bf16")


def grouped_sizes(groups=32, lo=64, hi=4096, seed=0):
    return [int(m) for m in rng(4, 99, seed).integers(lo, hi, size=groups, endpoint=True)]


def config4(groups=32, N=4096, K=2048, seed=0, m_sizes=None):
    """fp16 grouped GEMM, D_g = A_g.B_g + C_g, entries U[-1,1]."""
    ms = m_sizes if m_sizes is not None else grouped_sizes(groups, seed=seed)
    probs = []
    for g, m in enumerate(ms):
        A = uniform((m, K), -1, 1, "f16", 4, 3 * g + 0, seed)
        B = uniform((K, N), -1, 1, "f16", 4, 3 * g + 1, seed)
        C = uniform((m, N), -1, 1, "f16", 4, 3 * g + 2, seed)
        probs.append(Problem("fp16_grouped_g%d" % g, A, B, C, m, N, K, alpha=1.0, beta=1.0))
    return probs


def config4_e4m3(groups=32, N=4096, K=2048, seed=0, m_sizes=None):
    """The grouped shapes of config4 in fp8: e4m3 A_g, B_g ~ N(0,1) clamped to
    +-448, per-group per-tensor scales 2^U{-3..0}, bf16 out, beta 0."""
    ms = m_sizes if m_sizes is not None else grouped_sizes(groups, seed=seed)
    e = rng(4, 999, seed).integers(-3, 0, size=(len(ms), 2), endpoint=True)
    probs = []
    for g, m in enumerate(ms):
        A = normal((m, K), 1.0, "e4m3", 4, 1000 + 2 * g, seed)
        B = normal((K, N), 1.0, "e4m3", 4, 1001 + 2 * g, seed)
        probs.append(Problem("e4m3_grouped_g%d" % g, A, B, None, m, N, K, alpha=1.0, beta=0.0,
                             a_dtype="e4m3", b_dtype="e4m3", c_dtype="bf16", d_dtype="bf16",
                             scale_a=float(2.0 ** e[g, 0]), scale_b=float(2.0 ** e[g, 1])))
    return probs


def config5a(M, N, K, seed=0) -> Problem:
    """fp16 stream-K stress shape, entries U[-1,1], alpha = beta = 1."""
    wid = 5
    tid = 10 * STREAMK_SHAPES.index((M, N, K)) if (M, N, K) in STREAMK_SHAPES else 50 + (M + N + K) % 997
    A = uniform((M, K), -1, 1, "f16", wid, tid + 0, seed)
    B = uniform((K, N), -1, 1, "f16", wid, tid + 1, seed)
    C = uniform((M, N), -1, 1, "f16", wid, tid + 2, seed)
    return Problem("fp16_streamk_%dx%dx%d" % (M, N, K), A, B, C, M, N, K, alpha=1.0, beta=1.0)


def config5b(M=8192, N=8192, K=8192, scale_a=1.0, scale_b=1.0, seed=0) -> Problem:
    """e4m3 A, B ~ N(0,1) clamped to +-448, per-tensor fp32 scales, bf16 out, beta 0."""
    A = normal((M, K), 1.0, "e4m3", 5, 100, seed)
    B = normal((K, N), 1.0, "e4m3", 5, 101, seed)
    return Problem("e4m3_%dx%dx%d" % (M, N, K), A, B, None, M, N, K, alpha=1.0, beta=0.0,
                   a_dtype="e4m3", b_dtype="e4m3", c_dtype="bf16", d_dtype="bf16",
                   scale_a=scale_a, scale_b=scale_b)


# ---------------------------------------------------------------- block-scaled storage
#
# Element formats of the block-scaled GEMMs (MXFP8 / MXFP4 / NVFP4): the largest
# finite magnitude and the exponent of its leading bit (OCP MX element types).
MX_ELEMS = {"e4m3": (448.0, 8), "e5m2": (57344.0, 15), "e2m1": (6.0, 2)}
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_codes(x: np.ndarray) -> np.ndarray:
    """Nearest E2M1 code of each float64 value, ties to the even code,
    saturating at +-6; one code per byte, sign in bit 3 (negative zero kept)."""
    mag = np.minimum(np.abs(x), 6.0)
    lo = np.clip(np.searchsorted(E2M1_VALUES, mag, side="right") - 1, 0, 7)
    hi = np.minimum(lo + 1, 7)
    dlo, dhi = mag - E2M1_VALUES[lo], E2M1_VALUES[hi] - mag
    up = (dhi < dlo) | ((dhi == dlo) & (lo % 2 == 1))
    code = np.where(up, hi, lo).astype(np.uint8)
    return code | (np.signbit(x).astype(np.uint8) << 3)


def _elem_codes(x: np.ndarray, elem: str) -> np.ndarray:
    if elem == "e2m1":
        return e2m1_codes(x)
    mx = MX_ELEMS[elem][0]
    tdt = torch.float8_e4m3fn if elem == "e4m3" else torch.float8_e5m2
    # x is a float32 value times a power of two here: one rounding, saturating
    t = torch.from_numpy(np.clip(x, -mx, mx).astype(np.float32)).to(tdt)
    return t.view(torch.uint8).numpy()


def quantize_blocks(x: np.ndarray, elem: str, block: int, scale: str = "ue8m0", axis: int = 1):
    """Block-scaled storage of ``x`` (float32-representable values) with one
    scale per ``block`` consecutive entries along ``axis`` (the K axis: 1 for
    A [M, K], 0 for B [K, N]); a ragged last block is shorter.

    ``scale="ue8m0"`` (OCP MX): the block's scale is 2^X with
    X = floor(log2(amax)) - emax(elem), stored as the E8M0 code X + 127 (0 for
    an all-zero block); elements are x / 2^X rounded to nearest even in
    ``elem``, saturating.  ``scale="e4m3"`` (NVFP4 style): the scale is
    amax / max(elem) rounded to e4m3 (1 for an all-zero block) and the
    elements are x / scale rounded in ``elem``.

    Returns (element codes, same shape as x, uint8; scale codes, uint8, shape
    with ceil(K / block) along ``axis``)."""
    if scale == "e4m3" and elem != "e2m1":
        raise ValueError("e4m3 block scales go with e2m1 elements (NVFP4)")
    xt = np.moveaxis(np.asarray(x, dtype=np.float64), axis, -1)
    K = xt.shape[-1]
    kb = -(-K // block)
    pad = np.zeros(xt.shape[:-1] + (kb * block - K,))
    blocks = np.concatenate([xt, pad], axis=-1).reshape(xt.shape[:-1] + (kb, block))
    amax = np.abs(blocks).max(axis=-1)
    mx, emax = MX_ELEMS[elem]
    if scale == "ue8m0":
        with np.errstate(divide="ignore"):
            X = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - emax, -127)
        X = np.clip(X, -127, 127).astype(np.int64)
        s_codes = (X + 127).astype(np.uint8)
        s_val = np.ldexp(1.0, X)
    elif scale == "e4m3":
        s32 = torch.from_numpy(np.clip(amax / mx, 0, 448.0).astype(np.float32))
        s_codes = s32.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
        s_codes[s_codes == 0] = 0x38  # 1.0 for all-zero (or vanishing) blocks
        s_val = torch.from_numpy(s_codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    else:
        raise ValueError("scale must be 'ue8m0' or 'e4m3'")
    scaled = blocks / s_val[..., None]
    codes = _elem_codes(scaled, elem).reshape(blocks.shape[:-2] + (kb * block,))[..., :K]
    return np.moveaxis(codes, -1, axis).copy(), np.moveaxis(s_codes, -1, axis).copy()


def block_scaled_problem(M, N, K, elem="e4m3", block=32, scale="ue8m0", alpha=1.0, seed=0,
                         wid=11) -> Problem:
    """A seeded block-scaled GEMM: A [M, K] and B [K, N] drawn N(0, 1) (float32
    values) with a per-block magnitude spread of 2^U{-8..8}, quantised by
    ``quantize_blocks`` along K; row-major codes, bf16 output, beta 0.  The
    scale codes ride on the problem as ``block_scales = (SA, SB, scale, block)``."""
    key = (M * 1_000_003 + N * 10_007 + K * 101 + block) % (2 ** 31)
    g = rng(wid, key, seed)
    kb = -(-K // block)
    spread_a = np.repeat(np.ldexp(1.0, g.integers(-8, 9, size=(M, kb))), block, axis=1)[:, :K]
    spread_b = np.repeat(np.ldexp(1.0, g.integers(-8, 9, size=(kb, N))), block, axis=0)[:K]
    a = g.normal(0.0, 1.0, size=(M, K)).astype(np.float32).astype(np.float64) * spread_a
    b = g.normal(0.0, 1.0, size=(K, N)).astype(np.float32).astype(np.float64) * spread_b
    qa, sa = quantize_blocks(a, elem, block, scale, axis=1)
    qb, sb = quantize_blocks(b, elem, block, scale, axis=0)
    p = Problem("%s_%s_block%d_%dx%dx%d" % (elem, scale, block, M, N, K), torch.from_numpy(qa),
                torch.from_numpy(qb), None, M, N, K, alpha=alpha, beta=0.0, a_dtype=elem,
                b_dtype=elem, c_dtype="bf16", d_dtype="bf16")
    p.block_scales = (torch.from_numpy(sa), torch.from_numpy(sb), scale, block)
    return p


SCALE_ONE = {"ue8m0": 0x7F, "e4m3": 0x38}  # scale code of 1.0


def scale_atoms(codes: np.ndarray, one: int) -> np.ndarray:
    """Scale codes [R, SK] (R rows of a K-major operand, SK = K / block scales
    each, SK a multiple of 4) in the 128 x 4 blocked layout the tensor cores
    read: 512-byte atoms, atom (rb, cb) holding rows 128 rb .. 128 rb + 127 and
    scale columns 4 cb .. 4 cb + 3 at byte offset (rb * SK/4 + cb) * 512, the
    code of (r, c) at 16 * (r % 32) + 4 * ((r % 128) // 32) + c % 4 inside it.
    Rows past R up to the next multiple of 128 hold `one`."""
    R, SK = codes.shape
    if SK % 4:
        raise ValueError("the scale count along K must be a multiple of 4")
    RB = -(-R // 128)
    pad = np.full((RB * 128, SK), one, dtype=np.uint8)
    pad[:R] = codes
    t = pad.reshape(RB, 4, 32, SK // 4, 4)          # rb, q, i, cb, j with r = 128 rb + 32 q + i
    return np.ascontiguousarray(t.transpose(0, 3, 2, 1, 4)).reshape(-1)


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """E2M1 codes [R, K] (one per byte, low nibble) packed two per byte along
    K, element 2i in the low nibble: [R, K / 2]."""
    c = np.asarray(codes, dtype=np.uint8) & 0xF
    return np.ascontiguousarray(c[:, 0::2] | (c[:, 1::2] << 4))


def block_scaled_storage(prob):
    """The device storage of a block-scaled problem for the GEMM's TN layout:
    (A [M, K] codes, B as [N, K] codes (column-major B), SFA atoms, SFB atoms),
    fp4 codes packed two per byte; numpy uint8 arrays."""
    a = bits(prob.A)
    b = np.ascontiguousarray(bits(prob.B).T)
    sa, sb, scale, _ = prob.block_scales
    if prob.a_dtype == "e2m1":
        a, b = pack_e2m1(a), pack_e2m1(b)
    sfa = scale_atoms(bits(sa), SCALE_ONE[scale])
    sfb = scale_atoms(np.ascontiguousarray(bits(sb).T), SCALE_ONE[scale])
    return np.ascontiguousarray(a), b, sfa, sfb


def random_problem(M, N, K, dtype="f16", out_dtype=None, alpha=1.0, beta=0.0, relu=False,
                   a_col_major=False, b_col_major=False, seed=0, lo=-1.0, hi=1.0,
                   scale_a=1.0, scale_b=1.0, wid=9, act=None, bias=False,
                   aux_op=None) -> Problem:
    """A small seeded problem of any shape, layout and dtype, for edge-case tests
    (``bias=True`` adds a U[lo, hi] bias vector of N output-type elements;
    ``aux_op`` adds an M x N auxiliary tensor, U[0.5, 2] for "div" so that no
    divisor is near zero, U[lo, hi] otherwise)."""
    out_dtype = out_dtype or ("bf16" if dtype == "e4m3" else dtype)
    key = (M * 1_000_003 + N * 10_007 + K * 101 + int(a_col_major) * 2 + int(b_col_major)) % (2**31)
    sa, sb = _mk((M, K), (K, N), a_col_major, b_col_major)
    if dtype == "e4m3":
        A = normal(sa, 1.0, dtype, wid, key + 0, seed)
        B = normal(sb, 1.0, dtype, wid, key + 1, seed)
    else:
        A = uniform(sa, lo, hi, dtype, wid, key + 0, seed)
        B = uniform(sb, lo, hi, dtype, wid, key + 1, seed)
    C = uniform((M, N), lo, hi, out_dtype, wid, key + 2, seed) if beta != 0.0 else None
    bv = uniform((N,), lo, hi, out_dtype, wid, key + 3, seed) if bias else None
    zv = None
    if aux_op:
        zlo, zhi = (0.5, 2.0) if aux_op == "div" else (lo, hi)
        zv = uniform((M, N), zlo, zhi, out_dtype, wid, key + 4, seed)
    return Problem("random_%dx%dx%d" % (M, N, K), A, B, C, M, N, K, alpha=alpha, beta=beta,
                   relu=relu, a_dtype=dtype, b_dtype=dtype, c_dtype=out_dtype,
                   d_dtype=out_dtype, a_col_major=a_col_major, b_col_major=b_col_major,
                   scale_a=scale_a, scale_b=scale_b, act=act, bias=bv, aux=zv, aux_op=aux_op)


def integer_problem(M, N, K, dtype="f16", alpha=1.5, beta=0.5, act="relu",
                    a_col_major=False, b_col_major=False, seed=0, scale_a=1.0, scale_b=1.0,
                    bias=False, aux_op=None, wid=8) -> Problem:
    """A seeded problem whose GEMM arithmetic is exact in fp32: A and B hold
    integers in [-2, 2], C integers in [-4, 4], the bias integers in [-8, 8] and
    an auxiliary tensor integers in [-3, 3] (powers of two 1/2, 1, 2, 4 for
    "div").  With alpha, beta and the fp8 scales chosen so that every product
    is a short binary fraction, every partial sum, every epilogue step and the
    final value are exact in fp32, so that any k order gives the same result and
    the output is one round-to-nearest-even of the exact value: a GPU result is
    then comparable bit for bit with the oracle's rounded result."""
    out = "bf16" if dtype == "e4m3" else dtype
    key = (M * 1_000_003 + N * 10_007 + K * 101 + int(a_col_major) * 2 + int(b_col_major)) % (2**31)
    sa, sb = _mk((M, K), (K, N), a_col_major, b_col_major)
    A = integers(sa, -2, 2, dtype, wid, key + 0, seed)
    B = integers(sb, -2, 2, dtype, wid, key + 1, seed)
    C = integers((M, N), -4, 4, out, wid, key + 2, seed) if beta != 0.0 else None
    bv = integers((N,), -8, 8, out, wid, key + 3, seed) if bias else None
    zv = None
    if aux_op == "div":
        e = rng(wid, key + 4, seed).integers(-1, 2, size=(M, N), endpoint=True)
        zv = _store(np.ldexp(1.0, e), out)
    elif aux_op:
        zv = integers((M, N), -3, 3, out, wid, key + 4, seed)
    return Problem("int_%s_%dx%dx%d" % (dtype, M, N, K), A, B, C, M, N, K, alpha=alpha,
                   beta=beta, relu=act == "relu", a_dtype=dtype, b_dtype=dtype, c_dtype=out,
                   d_dtype=out, a_col_major=a_col_major, b_col_major=b_col_major,
                   scale_a=scale_a, scale_b=scale_b, act=act, bias=bv, aux=zv, aux_op=aux_op)

"""Pins of the CPU oracle against facts fixed outside it: the pages' worked
examples, closed forms, exact rational brute force on tiny inputs, library
decoders / rounding, and numpy's float64 matmul.  CPU only."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import check
from dense_gemm_15_gb300 import inputs
from conftest import read_golden

F16_ONE = 0x3C00


# ---------------------------------------------------------------- decoders

def test_decode_f16_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.decode(bits, "f16")
    ref = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(ours[m], ref[m])
    # signed zeros too
    assert np.array_equal(np.signbit(ours[m]), np.signbit(ref[m]))


def test_decode_bf16_all_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.decode(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(ours[m], ref[m])


def test_decode_e4m3_all_patterns_match_torch():
    bits = np.arange(256, dtype=np.uint8)
    ours = oracle.decode(bits, "e4m3")
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(ours[m], ref[m])
    assert np.nanmax(np.abs(ours)) == 448.0


# ---------------------------------------------------------------- rounding

def _f16_round_cases():
    g = np.random.default_rng(123)
    x = np.concatenate([
        g.standard_normal(20000) * np.exp2(g.integers(-30, 17, 20000)),
        # exact ties between neighbouring fp16 values
        (np.arange(0, 4096, dtype=np.float64) + 0.5) * 2.0 ** -24,
        (np.arange(1024, 2048, dtype=np.float64) + 0.5) * 2.0 ** -5,
        np.array([65504.0, 65519.0, 65519.999, 65520.0, 65536.0, 1e9,
                  2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0001, 2.0 ** -14,
                  2.0 ** -14 - 2.0 ** -25, 0.0, -0.0, 1025.0, 129.0]),
    ])
    return np.concatenate([x, -x])


def test_round_f16_matches_numpy():
    x = _f16_round_cases()
    ours = oracle.round_to(x, "f16")
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_round_bf16_matches_torch_on_float32_values():
    g = np.random.default_rng(7)
    x32 = (g.standard_normal(40000) * np.exp2(g.integers(-140, 127, 40000))).astype(np.float32)
    ties = ((np.arange(128, 256) + 0.5) * 2.0 ** -3).astype(np.float32)
    x32 = np.concatenate([x32, ties, -ties, np.float32([3.3895314e38, 0.0, -0.0])])
    ours = oracle.round_to(x32.astype(np.float64), "bf16")
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# ---------------------------------------------------------------- the pages' examples

@pytest.mark.parametrize("fixture", ["all_ones_128.txt", "all_ones_1024.txt"])
def test_all_ones_example(fixture):
    g = read_golden(fixture)
    M, N, K = (int(g[k][0][0]) for k in ("M", "N", "K"))
    a = np.full((M, K), F16_ONE, np.uint16)
    b = np.full((K, N), F16_ONE, np.uint16)
    c = np.full((M, N), F16_ONE, np.uint16)
    d = oracle.gemm(a, "f16", b, "f16", c, "f16", alpha=1.0, beta=1.0)
    assert np.all(d == float(g["expect_all"][0][0]))
    assert np.all(oracle.round_to(d, "f16") == int(g["expect_bits_all"][0][0], 16))


def test_alpha_beta_relu_hand_example():
    g = read_golden("alpha_beta_relu_2x2.txt")
    A = np.array([float(v) for v in g["A"][0]]).reshape(2, 2)
    B = np.array([float(v) for v in g["B"][0]]).reshape(2, 2)
    C = np.array([float(v) for v in g["C"][0]]).reshape(2, 2)
    f16 = lambda x: x.astype(np.float16).view(np.uint16)
    d = oracle.gemm(f16(A), "f16", f16(B), "f16", f16(C), "f16",
                    alpha=float(g["alpha"][0][0]), beta=float(g["beta"][0][0]),
                    relu=bool(int(g["relu"][0][0])))
    expect = np.array([float(v) for v in g["expect"][0]]).reshape(2, 2)
    assert np.array_equal(d, expect)


# ---------------------------------------------------------------- closed forms

def _rand_f16(shape, seed, lo=-1, hi=1):
    return np.random.default_rng(seed).uniform(lo, hi, shape).astype(np.float16).view(np.uint16)


def test_identity_b_returns_a():
    a = _rand_f16((37, 64), 1)
    eye = np.eye(64).astype(np.float16).view(np.uint16)
    d = oracle.gemm(a, "f16", eye, "f16")
    assert np.array_equal(oracle.round_to(d, "f16"), a)


def test_permutation_b_permutes_columns():
    a = _rand_f16((20, 48), 2)
    perm = np.random.default_rng(3).permutation(48)
    P = np.zeros((48, 48))
    P[perm, np.arange(48)] = 1.0  # column j of A.P is column perm[j] of A
    d = oracle.gemm(a, "f16", P.astype(np.float16).view(np.uint16), "f16")
    assert np.array_equal(oracle.round_to(d, "f16"), a[:, perm])


def test_rank1_outer_product():
    g = np.random.default_rng(4)
    u = g.integers(-4, 5, 24).astype(np.float64)
    v = g.integers(-4, 5, 40).astype(np.float64)
    K = 32
    A = np.repeat(u[:, None], K, axis=1)
    B = np.repeat(v[None, :], K, axis=0)
    d = oracle.gemm(A.astype(np.float16).view(np.uint16), "f16",
                    B.astype(np.float16).view(np.uint16), "f16")
    assert np.array_equal(d, K * np.outer(u, v))


def test_relu_of_negative_products_is_zero():
    a = np.full((16, 8), 0xBC00, np.uint16)  # -1
    b = np.full((8, 24), F16_ONE, np.uint16)
    c = np.zeros((16, 24), np.uint16)
    d = oracle.gemm(a, "f16", b, "f16", c, "f16", beta=1.0, relu=True)
    assert np.all(oracle.round_to(d, "f16") == 0)


def test_zero_a_gives_rounded_beta_c():
    c = _rand_f16((9, 33), 5, -10, 10)
    a = np.zeros((9, 7), np.uint16)
    b = _rand_f16((7, 33), 6)
    d = oracle.gemm(a, "f16", b, "f16", c, "f16", alpha=1.0, beta=0.5)
    want = (c.view(np.float16).astype(np.float64) * 0.5).astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.round_to(d, "f16"), want)


def test_alpha_beta_linearity_without_relu():
    p = inputs.random_problem(12, 20, 16, beta=1.0)
    a, b, c = inputs.bits(p.A), inputs.bits(p.B), inputs.bits(p.C)
    d1 = oracle.gemm(a, "f16", b, "f16", c, "f16", alpha=1.0, beta=0.0)
    d2 = oracle.gemm(a, "f16", b, "f16", c, "f16", alpha=0.0, beta=1.0)
    d3 = oracle.gemm(a, "f16", b, "f16", c, "f16", alpha=2.0, beta=-3.0)
    assert np.allclose(d3, 2.0 * d1 - 3.0 * d2, rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------------- exact brute force

def _exact_values(t: torch.Tensor):
    """Exact rationals of a stored CPU tensor, decoded by torch (not the oracle)."""
    return [[Fraction(float(v)) for v in row] for row in t.to(torch.float64).tolist()]


def _brute(p):
    A = _exact_values(p.A)
    B = _exact_values(p.B)
    C = _exact_values(p.C) if p.C is not None else None
    at = (lambda i, k: A[k][i]) if p.a_col_major else (lambda i, k: A[i][k])
    bt = (lambda k, j: B[j][k]) if p.b_col_major else (lambda k, j: B[k][j])
    s = Fraction(p.alpha) * Fraction(p.scale_a) * Fraction(p.scale_b)
    out = np.empty((p.M, p.N))
    mag = np.empty((p.M, p.N))
    for i in range(p.M):
        for j in range(p.N):
            acc = sum((at(i, k) * bt(k, j) for k in range(p.K)), Fraction(0))
            absacc = sum((abs(at(i, k) * bt(k, j)) for k in range(p.K)), Fraction(0))
            v = s * acc
            if p.beta != 0.0:
                v += Fraction(p.beta) * C[i][j]
            if p.relu and v < 0:
                v = Fraction(0)
            out[i, j] = float(v)
            mag[i, j] = float(abs(s) * absacc) + (abs(p.beta) * abs(float(C[i][j])) if p.beta else 0.0)
    return out, mag


def _oracle_of(p, **override):
    kw = dict(alpha=p.alpha, beta=p.beta, relu=p.relu, scale_a=p.scale_a, scale_b=p.scale_b,
              a_col_major=p.a_col_major, b_col_major=p.b_col_major)
    kw.update(override)
    return oracle.gemm(inputs.bits(p.A), p.a_dtype, inputs.bits(p.B), p.b_dtype,
                       inputs.bits(p.C) if p.C is not None else None, p.c_dtype, **kw)


def _agrees(d, exact, mag, K):
    return np.all(np.abs(d - exact) <= (K + 4) * 2.0 ** -52 * mag + 1e-300)


BRUTE_CASES = []
for dt in ("f16", "bf16", "e4m3"):
    for (M, N, K) in ((1, 1, 1), (3, 5, 7), (9, 9, 9), (4, 6, 2), (7, 3, 8)):
        for cm in ((False, False), (True, False), (False, True), (True, True)):
            BRUTE_CASES.append((dt, M, N, K, cm))


@pytest.mark.parametrize("dt,M,N,K,cm", BRUTE_CASES)
def test_brute_force_exact(dt, M, N, K, cm):
    p = inputs.random_problem(M, N, K, dtype=dt, alpha=1.5, beta=0.5 if dt != "e4m3" else -0.75,
                              relu=(M + N) % 2 == 0, a_col_major=cm[0], b_col_major=cm[1],
                              scale_a=0.37 if dt == "e4m3" else 1.0,
                              scale_b=1.7 if dt == "e4m3" else 1.0, lo=-3, hi=3)
    exact, mag = _brute(p)
    assert _agrees(_oracle_of(p), exact, mag, K)


def test_all_shapes_up_to_9():
    """Every M, N, K in 1..9 (with a subsample of combinations) against exact sums."""
    g = np.random.default_rng(11)
    for _ in range(60):
        M, N, K = (int(x) for x in g.integers(1, 10, 3))
        p = inputs.random_problem(M, N, K, beta=1.0, alpha=-2.0, seed=int(g.integers(1 << 30)))
        exact, mag = _brute(p)
        assert _agrees(_oracle_of(p), exact, mag, K)


# ------------------------------------------------- the pins catch planted mistakes

def test_planted_mistakes_are_caught():
    """Mistakes planted in the oracle's inputs or arithmetic (on the CPU) must
    fail the brute-force pin: a transposed operand, a dropped k term, a wrong
    sign of beta, ReLU applied before the beta*C add."""
    p = inputs.random_problem(6, 6, 6, beta=0.5, alpha=1.5, relu=True, lo=-3, hi=3)
    exact, mag = _brute(p)
    assert _agrees(_oracle_of(p), exact, mag, p.K)
    # transposed B (square, so the call is well formed)
    assert not _agrees(_oracle_of(p, b_col_major=True), exact, mag, p.K)
    # dropped last k term
    a, b = inputs.bits(p.A), inputs.bits(p.B)
    c = inputs.bits(p.C)
    dropped = oracle.gemm(np.ascontiguousarray(a[:, :-1]), "f16", np.ascontiguousarray(b[:-1]),
                          "f16", c, "f16", alpha=1.5, beta=0.5, relu=True)
    assert not _agrees(dropped, exact, mag, p.K)
    # wrong sign of beta
    assert not _agrees(_oracle_of(p, beta=-0.5), exact, mag, p.K)
    # ReLU before the beta*C add
    pre = oracle.gemm(a, "f16", b, "f16", alpha=1.5, relu=True)
    wrong = pre + 0.5 * oracle.decode(c, "f16")
    assert not _agrees(wrong, exact, mag, p.K)


# ---------------------------------------------------------------- bias and activations

def _f16i(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def test_bias_relu_example_exact():
    """kwkr.cn blog "CUTLASS Python接口" section 5.2: D = relu(A.B + bias), a bias
    of N elements added to every row, alpha 1, beta 0, at that section's shape
    M, N, K = 512, 1024, 768.  Small integer operands make every value exact;
    the expected result is integer numpy arithmetic.  A bias added along rows,
    or ReLU applied before the bias, would not match."""
    g = np.random.default_rng(11)
    M, N, K = 512, 1024, 768
    A = g.integers(-2, 3, (M, K))
    B = g.integers(-2, 3, (K, N))
    bias = g.integers(-60, 61, N)
    d = oracle.gemm(_f16i(A), "f16", _f16i(B), "f16", act="relu", bias=_f16i(bias))
    lin = A @ B
    assert np.array_equal(d, np.maximum(lin + bias[None, :], 0))
    # the data tell the plausible mistakes apart
    assert not np.array_equal(d, np.maximum(lin, 0) + bias[None, :])
    assert not np.array_equal(d[:, :M], np.maximum(lin[:, :M] + bias[:M, None], 0))


def test_bias_and_beta_c_are_both_added_before_the_activation():
    g = np.random.default_rng(12)
    A, B = g.integers(-3, 4, (7, 5)), g.integers(-3, 4, (5, 9))
    C, bias = g.integers(-8, 9, (7, 9)), g.integers(-8, 9, 9)
    d = oracle.gemm(_f16i(A), "f16", _f16i(B), "f16", _f16i(C), "f16", alpha=2.0, beta=-0.5,
                    act="relu", bias=_f16i(bias))
    assert np.array_equal(d, np.maximum(2.0 * (A @ B) - 0.5 * C + bias[None, :], 0))


def test_sigmoid_and_tanh_of_zero():
    """A zero product: sigmoid(0) = 1/2 and tanh(0) = 0 exactly."""
    a = np.zeros((6, 4), np.uint16)
    b = _rand_f16((4, 10), 13)
    assert np.array_equal(oracle.gemm(a, "f16", b, "f16", act="sigmoid"), np.full((6, 10), 0.5))
    assert np.array_equal(oracle.gemm(a, "f16", b, "f16", act="tanh"), np.zeros((6, 10)))


def test_sigmoid_and_tanh_match_library_routines():
    """Against scipy's logistic function and numpy's tanh applied to the
    oracle's own linear combination (with bias)."""
    from scipy.special import expit
    p = inputs.random_problem(24, 40, 32, beta=0.5, lo=-2, hi=2, bias=True)
    a, b, c, bv = (inputs.bits(t) for t in (p.A, p.B, p.C, p.bias))
    lin = oracle.gemm(a, "f16", b, "f16", c, "f16", alpha=1.5, beta=0.5, bias=bv)
    sig = oracle.gemm(a, "f16", b, "f16", c, "f16", alpha=1.5, beta=0.5, bias=bv, act="sigmoid")
    th = oracle.gemm(a, "f16", b, "f16", c, "f16", alpha=1.5, beta=0.5, bias=bv, act="tanh")
    assert np.allclose(sig, expit(lin), rtol=1e-14, atol=1e-15)
    assert np.allclose(th, np.tanh(lin), rtol=1e-14, atol=1e-15)
    assert np.all((sig >= 0) & (sig <= 1)) and np.all(np.abs(th) <= 1)


def test_tanh_is_twice_sigmoid_of_twice_minus_one():
    """tanh(x) = 2 sigmoid(2x) - 1 ties the two activations to each other:
    the same product with alpha doubled."""
    p = inputs.random_problem(16, 24, 20)
    a, b = inputs.bits(p.A), inputs.bits(p.B)
    th = oracle.gemm(a, "f16", b, "f16", alpha=0.75, act="tanh")
    sig2 = oracle.gemm(a, "f16", b, "f16", alpha=1.5, act="sigmoid")
    assert np.allclose(th, 2.0 * sig2 - 1.0, rtol=0, atol=1e-14)
    assert np.allclose(th, -oracle.gemm(a, "f16", b, "f16", alpha=-0.75, act="tanh"), atol=0)


@pytest.mark.parametrize("op", ["add", "sub", "mul", "div"])
def test_aux_tensor_ops_exact(op):
    """An auxiliary M x N tensor Z entering the activated value (the EFC
    operations of the CuteDSL page's roadmap section): small integer operands
    and power-of-two divisors keep every value exact; applying the operation
    before the activation would not match."""
    g = np.random.default_rng(21)
    A, B = g.integers(-3, 4, (9, 6)), g.integers(-3, 4, (6, 11))
    bias = g.integers(-5, 6, 11)
    Z = g.choice([-4.0, -2.0, -1.0, 1.0, 2.0, 4.0], (9, 11))
    d = oracle.gemm(_f16i(A), "f16", _f16i(B), "f16", act="relu", bias=_f16i(bias),
                    aux=_f16i(Z), aux_op=op)
    r = np.maximum(A @ B + bias[None, :], 0).astype(np.float64)
    want = {"add": r + Z, "sub": r - Z, "mul": r * Z, "div": r / Z}[op]
    assert np.array_equal(d, want)
    pre = (A @ B + bias[None, :]).astype(np.float64)
    wrong = np.maximum({"add": pre + Z, "sub": pre - Z, "mul": pre * Z, "div": pre / Z}[op], 0)
    assert not np.array_equal(d, wrong)


def test_aux_ops_invert_each_other():
    """(X * Z) / Z and (X / Z) * Z give X back exactly for Z = 2, and X - Z
    plus Z within the rounding of X - Z, with X the oracle's own result
    without Z."""
    p = inputs.random_problem(12, 20, 16, act="tanh", bias=True)
    a, b, bv = inputs.bits(p.A), inputs.bits(p.B), inputs.bits(p.bias)
    x = oracle.gemm(a, "f16", b, "f16", act="tanh", bias=bv)
    z = np.full((12, 20), 0x4000, np.uint16)  # 2.0
    assert np.array_equal(oracle.gemm(a, "f16", b, "f16", act="tanh", bias=bv, aux=z,
                                      aux_op="mul") / 2.0, x)
    assert np.array_equal(oracle.gemm(a, "f16", b, "f16", act="tanh", bias=bv, aux=z,
                                      aux_op="div") * 2.0, x)
    # x - 2 rounds to the spacing of numbers near 2: equal within that spacing
    assert np.allclose(oracle.gemm(a, "f16", b, "f16", act="tanh", bias=bv, aux=z,
                                   aux_op="sub") + 2.0, x, rtol=0, atol=2.0 ** -50)


# ---------------------------------------------------------------- block-scaled formats

def test_decode_e5m2_and_ue8m0_all_patterns_match_torch():
    bits = np.arange(256, dtype=np.uint8)
    for name, tdt in (("e5m2", torch.float8_e5m2), ("ue8m0", torch.float8_e8m0fnu)):
        ours = oracle.decode(bits, name)
        ref = torch.from_numpy(bits).view(tdt).to(torch.float64).numpy()
        assert np.array_equal(np.isnan(ours), np.isnan(ref)), name
        m = ~np.isnan(ref)
        assert np.array_equal(ours[m], ref[m]), name


def test_decode_e2m1_matches_the_format_table():
    """The 16 E2M1 codes: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 (OCP MX)."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    ours = oracle.decode(np.arange(16, dtype=np.uint8), "e2m1")
    assert list(ours[:8]) == mags and list(-ours[8:]) == mags
    assert np.all(np.signbit(ours[8:]))


def _mx_case(seed, M, N, K, block, elem):
    g = np.random.default_rng(seed)
    kb = -(-K // block)
    if elem == "e2m1":
        a = g.integers(0, 16, (M, K), dtype=np.uint8)
        b = g.integers(0, 16, (K, N), dtype=np.uint8)
    else:
        a = g.integers(0, 256, (M, K), dtype=np.uint8)
        b = g.integers(0, 256, (K, N), dtype=np.uint8)
        a[(a & 0x7F) == 0x7F] = 0x3C  # no NaN (e4m3) / keep finite
        b[(b & 0x7F) == 0x7F] = 0x3C
        if elem == "e5m2":
            a[(a & 0x7C) == 0x7C] = 0x3C  # no inf / NaN
            b[(b & 0x7C) == 0x7C] = 0x3C
    sa = g.integers(120, 135, (M, kb), dtype=np.uint8)
    sb = g.integers(120, 135, (kb, N), dtype=np.uint8)
    return a, b, sa, sb


@pytest.mark.parametrize("elem,block,K", [("e4m3", 32, 96), ("e5m2", 32, 80), ("e2m1", 32, 64),
                                          ("e2m1", 16, 40)])
def test_block_scaled_brute_force_exact(elem, block, K):
    """Block-scaled GEMM (MXFP8 / MXFP4 / NVFP4-style blocks) against exact
    rational arithmetic on values decoded by torch (e4m3, e5m2, E8M0) or the
    format table (e2m1); a scale indexed by k mod block instead of k / block
    fails."""
    M, N = 5, 7
    a, b, sa, sb = _mx_case(7, M, N, K, block, elem)
    tdt = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
    if elem == "e2m1":
        table = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6])
        av, bv = table[a], table[b]
    else:
        av = torch.from_numpy(a).view(tdt[elem]).to(torch.float64).numpy()
        bv = torch.from_numpy(b).view(tdt[elem]).to(torch.float64).numpy()
    sav = torch.from_numpy(sa).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    sbv = torch.from_numpy(sb).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    exact = np.zeros((M, N))
    wrong = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            acc = Fraction(0)
            bad = Fraction(0)
            for k in range(K):
                acc += Fraction(av[i, k]) * Fraction(sav[i, k // block]) * Fraction(bv[k, j]) * Fraction(sbv[k // block, j])
                kk = k % block if k % block < sav.shape[1] else 0
                bad += Fraction(av[i, k]) * Fraction(sav[i, kk]) * Fraction(bv[k, j]) * Fraction(sbv[kk, j])
            exact[i, j] = float(acc)
            wrong[i, j] = float(bad)
    d = oracle.gemm(a, elem, b, elem, scales=(sa, sb, "ue8m0", block))
    assert np.allclose(d, exact, rtol=1e-14, atol=0)
    assert not np.allclose(wrong, exact, rtol=1e-6, atol=0)


def test_unit_scales_equal_the_unscaled_product():
    """All E8M0 scales 127 (= 1): the block-scaled result is the plain one."""
    M, N, K = 8, 12, 64
    a, b, _, _ = _mx_case(3, M, N, K, 32, "e4m3")
    ones_a = np.full((M, 2), 127, np.uint8)
    ones_b = np.full((2, N), 127, np.uint8)
    assert np.array_equal(oracle.gemm(a, "e4m3", b, "e4m3", scales=(ones_a, ones_b, "ue8m0", 32)),
                          oracle.gemm(a, "e4m3", b, "e4m3"))


def test_nvfp4_blocks_with_e4m3_scales_and_tensor_scale():
    """NVFP4-style: E2M1 elements, E4M3 block scales per 16, a per-tensor scale
    as alpha; equals the plain product of operands pre-multiplied in float64."""
    M, N, K, block = 6, 10, 48, 16
    g = np.random.default_rng(5)
    a = g.integers(0, 16, (M, K), dtype=np.uint8)
    b = g.integers(0, 16, (K, N), dtype=np.uint8)
    sa = g.integers(0x30, 0x48, (M, K // block), dtype=np.uint8)  # positive finite e4m3
    sb = g.integers(0x30, 0x48, (K // block, N), dtype=np.uint8)
    d = oracle.gemm(a, "e2m1", b, "e2m1", alpha=0.25, scales=(sa, sb, "e4m3", block))
    av = oracle.decode(a, "e2m1") * np.repeat(oracle.decode(sa, "e4m3"), block, axis=1)
    bv = oracle.decode(b, "e2m1") * np.repeat(oracle.decode(sb, "e4m3"), block, axis=0)
    plain = oracle.gemm(np.ascontiguousarray(av), "f64", np.ascontiguousarray(bv), "f64", alpha=0.25)
    assert np.array_equal(d, plain)


# ---------------------------------------------------------------- cross-checks

def test_numpy_float64_cross_check():
    for dt in ("f16", "bf16"):
        p = inputs.random_problem(64, 96, 80, dtype=dt)
        d = _oracle_of(p)
        ref = p.A.to(torch.float64).numpy() @ p.B.to(torch.float64).numpy()
        assert np.allclose(d, ref, rtol=1e-12, atol=1e-12)


def test_row_sampling_and_thread_count_do_not_change_results():
    p = inputs.random_problem(40, 70, 33, beta=1.0, relu=True)
    a, b, c = inputs.bits(p.A), inputs.bits(p.B), inputs.bits(p.C)
    full1 = oracle.gemm(a, "f16", b, "f16", c, "f16", beta=1.0, relu=True, threads=1)
    full8 = oracle.gemm(a, "f16", b, "f16", c, "f16", beta=1.0, relu=True, threads=8)
    part = oracle.gemm(a, "f16", b, "f16", c, "f16", beta=1.0, relu=True, rows=(5, 17))
    assert np.array_equal(full1, full8)
    assert np.array_equal(part, full1[5:17])


def test_absolute_matches_abs_matmul():
    p = inputs.random_problem(30, 50, 40, dtype="bf16")
    ab = oracle.gemm(inputs.bits(p.A), "bf16", inputs.bits(p.B), "bf16", absolute=True)
    ref = np.abs(p.A.to(torch.float64).numpy()) @ np.abs(p.B.to(torch.float64).numpy())
    assert np.allclose(ab, ref, rtol=1e-12)


def test_beta_zero_never_reads_c():
    a = _rand_f16((4, 4), 8)
    d = oracle.gemm(a, "f16", a, "f16", None, "f16", beta=0.0)
    assert np.all(np.isfinite(d))


# ---------------------------------------------------------------- the checker

def test_checker_accepts_rounded_reference_and_rejects_perturbation():
    p = inputs.random_problem(32, 48, 64, beta=0.5, alpha=1.5, relu=True)
    d_ref, absab, c64 = check.reference(p, inputs.bits)
    bits = oracle.round_to(d_ref, "f16")
    ok, ratio, _, _ = check.compare(bits, "f16", d_ref, absab, c64, p)
    assert ok and ratio < 0.5
    bad = d_ref.copy()
    bad[3, 7] += 2.0 * check.bound(absab, p.alpha, p.beta, c64, "f16")[3, 7] + 0.01
    ok, ratio, idx, nbad = check.compare(oracle.round_to(bad, "f16"), "f16", d_ref, absab, c64, p)
    assert not ok and nbad == 1 and tuple(idx) == (3, 7)

"""The seeded block-scaled input generator on CPU: E2M1 rounding against brute
force, the E8M0 / E4M3 scale choice and the quantisation error of every
element against the element format's half-unit in the last place, and a
generated problem through the oracle against a float64 product of operands
decoded by torch (or the E2M1 table), not by the oracle."""
import numpy as np
import pytest
import torch

import oracle
from dense_gemm_15_gb300 import inputs as I
from oracle import check

# mantissa bits, smallest normal exponent, largest magnitude
FORMATS = {"e4m3": (3, -6, 448.0), "e5m2": (2, -14, 57344.0), "e2m1": (1, 0, 6.0)}
TABLE = np.concatenate([I.E2M1_VALUES, -I.E2M1_VALUES])


def _decode_elem(codes, elem):
    if elem == "e2m1":
        return TABLE[codes & 0xF]  # codes 8..15 are the negatives
    tdt = torch.float8_e4m3fn if elem == "e4m3" else torch.float8_e5m2
    return torch.from_numpy(np.ascontiguousarray(codes)).view(tdt).to(torch.float64).numpy()


def _decode_scale(codes, scale):
    tdt = torch.float8_e8m0fnu if scale == "ue8m0" else torch.float8_e4m3fn
    return torch.from_numpy(np.ascontiguousarray(codes)).view(tdt).to(torch.float64).numpy()


def _half_ulp(v, elem):
    m, emin, _ = FORMATS[elem]
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** (emin - 1))))
    return np.ldexp(0.5, (np.maximum(e, emin) - m).astype(int))


def test_e2m1_rounding_matches_brute_force():
    x = np.concatenate([np.arange(-7.0, 7.0001, 0.125), [0.0, -0.0, 1e-9, 100.0, -100.0]])
    codes = I.e2m1_codes(x)
    for v, c in zip(x, codes):
        mag = min(abs(v), 6.0)
        d = np.abs(I.E2M1_VALUES - mag)
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [i for i in best if i % 2 == 0][0]
        assert c & 0x7 == want, (v, c)
        assert (c >> 3) == int(np.signbit(v)), (v, c)


def _raw(shape, seed):
    g = np.random.default_rng(seed)
    x = g.normal(0, 1, size=shape).astype(np.float32).astype(np.float64)
    return x * np.ldexp(1.0, g.integers(-8, 9, size=shape))


@pytest.mark.parametrize("elem,block,scale,axis", [
    ("e4m3", 32, "ue8m0", 1), ("e5m2", 32, "ue8m0", 0), ("e2m1", 32, "ue8m0", 1),
    ("e2m1", 16, "e4m3", 0), ("e4m3", 32, "ue8m0", 0)])
def test_quantised_blocks_are_within_half_an_ulp(elem, block, scale, axis):
    K = 3 * block + 5  # ragged last block
    shape = (K, 24) if axis == 0 else (24, K)
    x = _raw(shape, 3)
    if axis:
        x[1, :block] = 0.0  # an all-zero block
    else:
        x[:block, 1] = 0.0
    q, s = I.quantize_blocks(x, elem, block, scale, axis=axis)
    kb = -(-K // block)
    assert q.shape == x.shape and s.shape == ((kb, 24) if axis == 0 else (24, kb))
    sv = _decode_scale(s, scale)
    sv_full = np.repeat(sv, block, axis=axis)[(slice(None), slice(0, K)) if axis else slice(0, K)]
    scaled = x / sv_full
    back = _decode_elem(q, elem)
    mx = FORMATS[elem][2]
    sat = np.abs(scaled) > mx
    assert np.all(np.abs(back[sat]) == mx)
    err = np.abs(back - scaled)[~sat]
    assert np.all(err <= _half_ulp(scaled[~sat], elem)), err.max()
    # scale choice: the block maximum lands in the top binade of the element format
    xt = np.moveaxis(x, axis, -1)
    pad = np.zeros(xt.shape[:-1] + (kb * block - K,))
    amax = np.abs(np.concatenate([xt, pad], -1).reshape(xt.shape[:-1] + (kb, block))).max(-1)
    svt = np.moveaxis(sv, axis, -1)
    nz = amax > 0
    if scale == "ue8m0":
        emax = I.MX_ELEMS[elem][1]
        r = amax[nz] / svt[nz]
        assert np.all((r >= 2.0 ** emax) & (r < 2.0 ** (emax + 1)))
        assert np.all(np.moveaxis(s, axis, -1)[~nz] == 0)
    else:
        # e4m3 scale = amax / 6 rounded to e4m3 (relative half-ulp 2^-4 in its normal range)
        assert np.all(np.abs(svt[nz] - amax[nz] / 6.0) <= 2.0 ** -4 * amax[nz] / 6.0 + 2.0 ** -10)
        assert np.all(svt[~nz] == 1.0)


def test_e4m3_scales_need_e2m1_elements():
    with pytest.raises(ValueError):
        I.quantize_blocks(np.ones((2, 32)), "e4m3", 32, "e4m3")


@pytest.mark.parametrize("elem,block,scale", [("e4m3", 32, "ue8m0"), ("e5m2", 32, "ue8m0"),
                                              ("e2m1", 32, "ue8m0"), ("e2m1", 16, "e4m3")])
def test_block_scaled_problem_through_the_oracle(elem, block, scale):
    p = I.block_scaled_problem(20, 40, 2 * block + 8, elem, block, scale, alpha=0.5)
    sa, sb, sdt, blk = p.block_scales
    assert sdt == scale and blk == block
    a = _decode_elem(p.A.numpy(), elem) * np.repeat(_decode_scale(sa.numpy(), scale), block, 1)[:, :p.K]
    b = _decode_elem(p.B.numpy(), elem) * np.repeat(_decode_scale(sb.numpy(), scale), block, 0)[:p.K]
    want = 0.5 * (a @ b)
    d_ref, absab, c64 = check.reference(p, I.bits)
    assert c64 is None
    assert np.allclose(d_ref, want, rtol=1e-12, atol=1e-300)
    assert np.allclose(absab, np.abs(a) @ np.abs(b), rtol=1e-12, atol=1e-300)
    # a check of the rounded result passes, one with a scale block dropped fails
    d16 = oracle.round_to(d_ref, "bf16")
    assert check.compare(d16, "bf16", d_ref, absab, c64, p)[0]
    p.block_scales = (sa, sb.clone().fill_(127 if scale == "ue8m0" else 0x38), sdt, blk)
    d_bad, _, _ = check.reference(p, I.bits)
    assert not check.compare(oracle.round_to(d_bad, "bf16"), "bf16", d_ref, absab, c64, p)[0]


def test_integer_problems_are_exact_in_fp32():
    """The small-integer problems of the bit-exact GPU tests: the oracle's
    result equals exact integer arithmetic (numpy int64 on the decoded
    operands, scaled by alpha, beta and the fp8 scales as exact fractions),
    and every magnitude the GPU forms (the k sums, alpha * sum, the epilogue
    terms) stays below 2^24, so fp32 holds each of them exactly."""
    from fractions import Fraction
    import oracle
    for dtype, kw in (("f16", dict(bias=True, aux_op="mul")), ("bf16", dict(aux_op="div")),
                      ("e4m3", dict(beta=0.0, scale_a=0.5, scale_b=0.25, bias=True))):
        p = I.integer_problem(24, 40, 4224, dtype=dtype, act="linear", **kw)
        a = p.A.double().numpy().astype(np.int64)
        b = p.B.double().numpy().astype(np.int64)
        assert np.abs(a).max() <= 2 and np.abs(b).max() <= 2
        s = a @ b
        assert np.abs(s).max() * 4 < 2 ** 24
        alpha = Fraction(p.alpha) * Fraction(p.scale_a) * Fraction(p.scale_b)
        want = s.astype(object) * alpha
        if p.beta != 0.0:
            want = want + p.C.double().numpy().astype(np.int64).astype(object) * Fraction(p.beta)
        if p.bias is not None:
            want = want + p.bias.double().numpy().astype(np.int64).astype(object)[None, :]
        if p.aux_op == "mul":
            want = want * p.aux.double().numpy().astype(np.int64).astype(object)
        elif p.aux_op == "div":
            z = p.aux.double().numpy()
            assert set(np.unique(z)) <= {0.5, 1.0, 2.0, 4.0}
            want = want / np.vectorize(Fraction)(z).astype(object)
        got = oracle.gemm(I.bits(p.A), p.a_dtype, I.bits(p.B), p.b_dtype,
                          I.bits(p.C) if p.C is not None else None, p.c_dtype,
                          alpha=p.alpha, beta=p.beta, scale_a=p.scale_a, scale_b=p.scale_b,
                          bias=I.bits(p.bias) if p.bias is not None else None,
                          bias_dtype=p.d_dtype,
                          aux=I.bits(p.aux) if p.aux_op else None, aux_dtype=p.d_dtype,
                          aux_op=p.aux_op)
        assert all(Fraction(float(x)) == y for x, y in zip(got.ravel(), want.ravel()))
        assert max(abs(float(y)) for y in want.ravel()) < 2 ** 23


def test_scale_atoms_and_fp4_packing_place_every_code():
    """The blocked scale layout and the fp4 packing, checked element by
    element against their definitions (storage only: no arithmetic)."""
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 255, size=(200, 12)).astype(np.uint8)
    at = I.scale_atoms(codes, 0x7F)
    assert at.size == 2 * 3 * 512
    for r in range(256):
        for c in range(12):
            off = (r // 128 * 3 + c // 4) * 512 + 16 * (r % 32) + 4 * ((r % 128) // 32) + c % 4
            assert at[off] == (codes[r, c] if r < 200 else 0x7F)
    q = rng.integers(0, 16, size=(3, 10)).astype(np.uint8)
    pk = I.pack_e2m1(q)
    assert pk.shape == (3, 5)
    assert np.array_equal(pk & 0xF, q[:, 0::2]) and np.array_equal(pk >> 4, q[:, 1::2])
    with pytest.raises(ValueError):
        I.scale_atoms(codes[:, :6], 0x7F)

"""Comparison of a GPU result against the oracle -- test infrastructure only.

Tolerance for fp16 / bf16 output (element by element):

    |D - D_ref| <= 1e-2 * |alpha| * s_a * s_b * (|A| . |B|)_ij + 1e-3
                   + u * (|beta * C_ij| + |bias_j|)
                   [+ u * |D_ref_ij| for sigmoid and tanh]

and, with an auxiliary tensor Z entering after the activation, that bound E
becomes E + u*(|Z| + |D_ref|) for add / sub, E*|Z| + u*|D_ref| for mul and
E/|Z| + u*|D_ref| for div (the error of the activated value carried through
the operation, plus one rounding of the result).

with u = 2^-10 for fp16 and 2^-7 for bf16 output.  The first two terms are the
stated bound of the method's accuracy target; |alpha| and s_a*s_b scale it
with the product term it bounds (for alpha = s = 1 it is the literal bound),
and the u terms cover the one rounding of the result to the output type
where the relative term does not: the beta*C and bias contributions, and the
value of a bounded activation (sigmoid, tanh), which need not be small where
|A|.|B| is.  ReLU, sigmoid (1/4) and tanh are 1-Lipschitz, so the bound on the
linear combination holds after them.
"""
from __future__ import annotations

import numpy as np

from . import decode, gemm

ROUND_UNIT = {"f16": 2.0 ** -10, "bf16": 2.0 ** -7}


def bound(absab: np.ndarray, alpha: float, beta: float, c64, out_dtype: str,
          scale=1.0, bias64=None, d_ref=None) -> np.ndarray:
    b = 1e-2 * abs(alpha) * scale * absab + 1e-3
    if beta != 0.0 and c64 is not None:
        b = b + ROUND_UNIT[out_dtype] * np.abs(beta * c64)
    if bias64 is not None:
        b = b + ROUND_UNIT[out_dtype] * np.abs(bias64)[None, :]
    if d_ref is not None:
        b = b + ROUND_UNIT[out_dtype] * np.abs(np.nan_to_num(d_ref))
    return b


def _act(prob):
    return getattr(prob, "act", None) or ("relu" if prob.relu else "linear")


def reference(prob, bits_of, rows=None, threads=None):
    """(D_ref, |A|.|B|, C as float64) for rows ``rows`` of ``prob``.

    ``bits_of`` maps a CPU tensor to its stored bits (the input module's
    ``bits``), so this module needs nothing from the CUDA path."""
    a, b = bits_of(prob.A), bits_of(prob.B)
    c = bits_of(prob.C) if prob.C is not None else None
    scales = getattr(prob, "block_scales", None)
    if scales is not None:
        scales = (bits_of(scales[0]), bits_of(scales[1]), scales[2], scales[3])
    bias = getattr(prob, "bias", None)
    aux_op = getattr(prob, "aux_op", None)
    aux = bits_of(prob.aux) if aux_op else None
    d_ref = gemm(a, prob.a_dtype, b, prob.b_dtype, c if prob.beta != 0.0 else None,
                 prob.c_dtype, alpha=prob.alpha, beta=prob.beta, act=_act(prob),
                 bias=bits_of(bias) if bias is not None else None, bias_dtype=prob.d_dtype,
                 aux=aux, aux_dtype=prob.d_dtype, aux_op=aux_op,
                 scale_a=prob.scale_a, scale_b=prob.scale_b,
                 a_col_major=prob.a_col_major, b_col_major=prob.b_col_major,
                 rows=rows, threads=threads, scales=scales)
    absab = gemm(a, prob.a_dtype, b, prob.b_dtype, absolute=True,
                 a_col_major=prob.a_col_major, b_col_major=prob.b_col_major,
                 rows=rows, threads=threads, scales=scales)
    c64 = None
    if c is not None and prob.beta != 0.0:
        r0, r1 = (0, prob.M) if rows is None else rows
        c64 = decode(c[r0:r1], prob.c_dtype)
    return d_ref, absab, c64


def _bits16(t):
    """Stored bits of a 16-bit CPU tensor (without importing the input module)."""
    import torch
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def compare(d_bits: np.ndarray, out_dtype: str, d_ref, absab, c64, prob):
    """Returns (ok, worst ratio |err|/bound, index of worst, count of failures)."""
    d = decode(d_bits, out_dtype)
    bias = getattr(prob, "bias", None)
    bias64 = decode(bias.view(np.uint16) if isinstance(bias, np.ndarray) else _bits16(bias),
                    out_dtype) if bias is not None else None
    tol = bound(absab, prob.alpha, prob.beta, c64, out_dtype, prob.scale_a * prob.scale_b,
                bias64=bias64, d_ref=d_ref if _act(prob) in ("sigmoid", "tanh") else None)
    aux_op = getattr(prob, "aux_op", None)
    if aux_op:
        z = _bits16(prob.aux)
        if d_ref.shape[0] != prob.M:
            raise ValueError("aux checks compare whole results")
        z64 = np.abs(decode(z, out_dtype))
        u = ROUND_UNIT[out_dtype]
        dr = u * np.abs(np.nan_to_num(d_ref))
        if aux_op in ("add", "sub"):
            tol = tol + u * z64 + dr
        elif aux_op == "mul":
            tol = tol * z64 + dr
        else:
            tol = tol / z64 + dr
    err = np.abs(d - d_ref)
    ratio = np.where(np.isfinite(err), err / tol, np.inf)
    # NaN where the reference is NaN too counts as agreement.
    both_nan = np.isnan(d) & np.isnan(d_ref)
    ratio = np.where(both_nan, 0.0, ratio)
    if ratio.size == 0:
        return True, 0.0, None, 0
    worst = int(np.argmax(ratio))
    nbad = int(np.count_nonzero(ratio > 1.0))
    return nbad == 0, float(ratio.flat[worst]), np.unravel_index(worst, ratio.shape), nbad

"""Dense and grouped block-scaled GEMM with their epilogues (oracle; test infrastructure).

Dense ("GEMM + Amax (SM100)", Equations):
    C[m, n, l] = sum_k Ahat[m, k, l] * Bhat[n, k, l],   Amax = max |C|.

Grouped ("Grouped GEMM + sReLU (SM100)", Equations and Tanh soft clamp; the row
ranges as defined by "Grouped GEMM (SM100 BF16)", Operation): rows
[padded_offsets[g-1], padded_offsets[g]) (0 for g = 0) belong to expert g, and

    C[m, n] = alpha_g * sum_k Ahat[m, k] * Bhat[n, k, g]
    D[m, n] = prob[m] * relu(C[m, n])^2                      (no clamp)
    D[m, n] = prob[m] * (s * min(tanh(relu(C[m, n]) / s), 1))^2  (tanh_clamp_scale s)
    Amax[g] = max over the rows of g of |D|   (0 for an expert with no rows).

FP8 D ("Grouped GEMM + sReLU (SM100)", Shapes: SFD_row per 32 columns, SFD_col per
32 rows; the quantisation formula of "Grouped GEMM + dSwiGLU (SM100)", Step 3):
the scale of a block is norm_const * blockamax(|D|) / 448 rounded up to a power of
two (E8M0), and the stored code is RNE_satfinite_E4M3(D * norm_const / scale).
D_row uses blocks of 32 consecutive columns of a row, D_col blocks of 32
consecutive rows of a column; both are stored (valid_m, N) row-major.

Everything is float64; the matrix products use numpy's matmul as the library
primitive.  Results are unrounded unless a function says otherwise.
"""
from __future__ import annotations

import numpy as np

from . import formats, quantize, sf_layout


def dense_gemm_amax(a_codes, b_codes, sfa, sfb, fmt: str, m: int, n: int, k: int, l: int):
    """Returns (C float64 (L, M, N), amax float64)."""
    ahat = quantize.dequantize(a_codes, sfa, fmt, m, k, l)
    bhat = quantize.dequantize(b_codes, sfb, fmt, n, k, l)
    c = np.matmul(ahat, np.swapaxes(bhat, -1, -2))
    return c, float(np.max(np.abs(c))) if c.size else 0.0


def dense_abs_sum(a_codes, b_codes, sfa, sfb, fmt, m, n, k, l):
    """sum_k |Ahat||Bhat| per output element (the scale of the accumulation error bound)."""
    ahat = np.abs(quantize.dequantize(a_codes, sfa, fmt, m, k, l))
    bhat = np.abs(quantize.dequantize(b_codes, sfb, fmt, n, k, l))
    return np.matmul(ahat, np.swapaxes(bhat, -1, -2))


def expert_of_rows(padded_offsets, valid_m: int) -> np.ndarray:
    """Expert id of every row in [0, valid_m)."""
    ends = np.asarray(padded_offsets, dtype=np.int64)
    begin = 0
    g_of = np.full(valid_m, -1, dtype=np.int64)
    for g, end in enumerate(ends):
        g_of[begin:end] = g
        begin = end
    return g_of


def srelu(c, prob, tanh_clamp_scale=None):
    """D from C (float64): prob * relu(C)^2, or prob * (s * min(tanh(relu(C)/s), 1))^2."""
    r = np.maximum(c, 0.0)
    if tanh_clamp_scale is not None:
        s = float(tanh_clamp_scale)
        r = s * np.minimum(np.tanh(r / s), 1.0)
    return np.asarray(prob, dtype=np.float64).reshape(-1, 1) * (r * r)


def grouped_gemm(a_codes, b_codes, sfa, sfb, fmt: str, padded_offsets, alpha, k: int, n: int):
    """C float64 (valid_m, N) = alpha_g * Ahat_rows(g) @ Bhat[g]^T over each expert's rows."""
    ends = np.asarray(padded_offsets, dtype=np.int64)
    num_experts = len(ends)
    valid_m = int(ends[-1])
    ahat = quantize.dequantize(a_codes, sfa, fmt, valid_m, k, 1)[0]
    bhat = quantize.dequantize(b_codes, sfb, fmt, n, k, num_experts)
    c = np.zeros((valid_m, n), dtype=np.float64)
    begin = 0
    for g in range(num_experts):
        end = int(ends[g])
        if end > begin:
            c[begin:end] = float(alpha[g]) * (ahat[begin:end] @ bhat[g].T)
        begin = end
    return c


def per_expert_amax(d, padded_offsets) -> np.ndarray:
    ends = np.asarray(padded_offsets, dtype=np.int64)
    out = np.zeros(len(ends), dtype=np.float64)
    begin = 0
    for g, end in enumerate(ends):
        if end > begin:
            out[g] = np.max(np.abs(d[begin:end]))
        begin = end
    return out


def mxfp8_quantize_blocks(d, norm_const: float, axis: int):
    """Quantise D (rows, cols) in blocks of 32 along ``axis`` (1: rows of 32 columns, 0: columns).

    Returns (codes uint8 same shape as D, scale codes logical (rows, cols/32) for
    axis 1 or (cols, rows/32) for axis 0).
    """
    d = np.asarray(d, dtype=np.float64)
    x = d if axis == 1 else d.T
    r, c = x.shape
    xb = x.reshape(r, c // 32, 32)
    amax = np.abs(xb).max(axis=-1)
    sf = formats.e8m0_ceil_code(float(norm_const) * amax)
    scale = formats.decode_e8m0(sf)
    codes = formats.encode_e4m3(xb * float(norm_const) / scale[..., None]).reshape(r, c)
    return (codes if axis == 1 else codes.T.copy()), sf


def grouped_srelu(a_codes, b_codes, sfa, sfb, fmt: str, padded_offsets, alpha, prob, k: int, n: int,
                  tanh_clamp_scale=None, d_fp8: bool = False, norm_const: float = 1.0):
    """The whole grouped path.  Returns a dict with float64 C, D, amax (L,) and, for
    FP8 D, codes d_row / d_col and the physical SFD_row / SFD_col buffers."""
    c = grouped_gemm(a_codes, b_codes, sfa, sfb, fmt, padded_offsets, alpha, k, n)
    d = srelu(c, prob, tanh_clamp_scale)
    out = {"c": c, "d": d, "amax": per_expert_amax(d, padded_offsets)}
    if d_fp8:
        valid_m = c.shape[0]
        d_row, sf_row = mxfp8_quantize_blocks(d, norm_const, axis=1)
        d_col, sf_col = mxfp8_quantize_blocks(d, norm_const, axis=0)
        out.update(d_row=d_row, d_col=d_col,
                   sfd_row=sf_layout.pack(sf_row[None]), sfd_col=sf_layout.pack(sf_col[None]),
                   sfd_row_logical=sf_row, sfd_col_logical=sf_col)
        assert sf_row.shape == (valid_m, n // 32) and sf_col.shape == (n, valid_m // 32)
    return out

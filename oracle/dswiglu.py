"""Grouped block-scaled GEMM + dSwiGLU backward epilogue (oracle; test infrastructure).

"Grouped GEMM + dSwiGLU (SM100)", Shapes, Equations (Steps 1-3) and Diagram.  Rows
[padded_offsets[g-1], padded_offsets[g]) belong to expert g (as in the grouped GEMM
pages).  With the forward intermediate C of 2N columns, beta_g its per-expert scale
and prob the per-row gate:

    ref[m, n]  = alpha_g * sum_k Ahat[m, k] * Bhat[n, k, g]            (Step 1)
    x, gate    = the input and gate halves of beta_g * C[m, :]           (Step 2)
    sig        = 1 / (1 + exp(-gate)),   swish = gate * sig
    ab         = ref * prob * swish
    dswiglu    = ref * prob * x * sig * (1 + gate * (1 - sig))
    dprob[m]  += sum_n swish * x * ref
    D          = ab and dswiglu interleaved back into 2N columns
    amax[g]    = (max |ab|, max |dswiglu|) over the rows of expert g    (bf16 / f16 / f32 D)
    FP8 D: row and column MXFP8 quantisation of D as for the grouped sReLU D (Step 3).

Readings of the page taken here (each also listed in the design notes):
* Step 1 prints alpha_g squared, while the page's diagram applies alpha[group_idx] once
  and the grouped sReLU page scales by alpha_g: ref uses alpha_g once.  (A caller that
  wants alpha_g squared passes the squares.)
* "32-column interleaving along 2N": the 2N columns are 32-wide blocks alternating
  input, gate, input, gate, ...; ref column n (block j = n // 32, offset i = n % 32)
  pairs with input column 64 j + i and gate column 64 j + 32 + i, and D puts ab and
  dswiglu at the same two columns.  N is a multiple of 32.
* amax has shape (L, 2): column 0 is the maximum of |ab| (the input-gradient blocks),
  column 1 of |dswiglu| (the gate-gradient blocks); 0 for an expert without rows.
* dprob is accumulated into the caller's (zero-initialised) buffer: the page's sum over
  32-column chunks equals the sum over all N columns in exact arithmetic.

Everything is float64; results are unrounded unless a function says otherwise.
"""
from __future__ import annotations

import numpy as np

from . import gemm, sf_layout

BLOCK = 32


def deinterleave(c2) -> tuple[np.ndarray, np.ndarray]:
    """(rows, 2N) -> (input (rows, N), gate (rows, N)) by alternating 32-column blocks."""
    c2 = np.asarray(c2, dtype=np.float64)
    rows, two_n = c2.shape
    assert two_n % (2 * BLOCK) == 0
    blocks = c2.reshape(rows, two_n // (2 * BLOCK), 2, BLOCK)
    n = two_n // 2
    return blocks[:, :, 0, :].reshape(rows, n), blocks[:, :, 1, :].reshape(rows, n)


def interleave(x, y) -> np.ndarray:
    """Inverse of ``deinterleave``: 32-column blocks of x and y alternate, x first."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    rows, n = x.shape
    assert y.shape == x.shape and n % BLOCK == 0
    out = np.empty((rows, n // BLOCK, 2, BLOCK), dtype=np.float64)
    out[:, :, 0, :] = x.reshape(rows, n // BLOCK, BLOCK)
    out[:, :, 1, :] = y.reshape(rows, n // BLOCK, BLOCK)
    return out.reshape(rows, 2 * n)


def sigmoid(g) -> np.ndarray:
    """1 / (1 + exp(-g)) without overflow for large |g|."""
    g = np.asarray(g, dtype=np.float64)
    e = np.exp(-np.abs(g))
    return np.where(g >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def epilogue(ref, x, gate, prob):
    """Step 2 on already-scaled halves: returns (ab, dswiglu, dprob (rows,))."""
    ref = np.asarray(ref, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    gate = np.asarray(gate, dtype=np.float64)
    p = np.asarray(prob, dtype=np.float64).reshape(-1, 1)
    sig = sigmoid(gate)
    swish = gate * sig
    ab = ref * p * swish
    dsw = ref * p * x * sig * (1.0 + gate * (1.0 - sig))
    dprob = np.sum(swish * x * ref, axis=1)
    return ab, dsw, dprob


def per_expert_amax2(ab, dsw, padded_offsets) -> np.ndarray:
    """(L, 2): max |ab| and max |dswiglu| over each expert's rows (0 if it has none)."""
    ends = np.asarray(padded_offsets, dtype=np.int64)
    out = np.zeros((len(ends), 2), dtype=np.float64)
    begin = 0
    for g, end in enumerate(ends):
        if end > begin:
            out[g, 0] = np.max(np.abs(ab[begin:end]))
            out[g, 1] = np.max(np.abs(dsw[begin:end]))
        begin = end
    return out


def grouped_dswiglu(a_codes, b_codes, sfa, sfb, fmt: str, padded_offsets, alpha, beta, prob, c_in,
                    k: int, n: int, d_fp8: bool = False, norm_const: float = 1.0):
    """The whole grouped dSwiGLU path.  ``c_in`` (valid_m, 2N) holds the values of the stored
    forward intermediate (exactly as stored, e.g. bf16 values).  Returns a dict with float64
    ref, ab, dswiglu, D (valid_m, 2N), dprob (valid_m,), amax (L, 2) and, for FP8 D, codes
    d_row / d_col and the physical SFD_row / SFD_col buffers (2N columns)."""
    ref = gemm.grouped_gemm(a_codes, b_codes, sfa, sfb, fmt, padded_offsets, alpha, k, n)
    valid_m = ref.shape[0]
    g_of = gemm.expert_of_rows(padded_offsets, valid_m)
    beta_rows = np.asarray(beta, dtype=np.float64)[np.maximum(g_of, 0)].reshape(-1, 1)
    x, gate = deinterleave(np.asarray(c_in, dtype=np.float64) * beta_rows)
    ab, dsw, dprob = epilogue(ref, x, gate, prob)
    d = interleave(ab, dsw)
    out = {"ref": ref, "ab": ab, "dswiglu": dsw, "d": d, "dprob": dprob,
           "amax": per_expert_amax2(ab, dsw, padded_offsets), "x": x, "gate": gate}
    if d_fp8:
        d_row, sf_row = gemm.mxfp8_quantize_blocks(d, norm_const, axis=1)
        d_col, sf_col = gemm.mxfp8_quantize_blocks(d, norm_const, axis=0)
        out.update(d_row=d_row, d_col=d_col,
                   sfd_row=sf_layout.pack(sf_row[None]), sfd_col=sf_layout.pack(sf_col[None]),
                   sfd_row_logical=sf_row, sfd_col_logical=sf_col)
        assert sf_row.shape == (valid_m, 2 * n // 32) and sf_col.shape == (2 * n, valid_m // 32)
    return out

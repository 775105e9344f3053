"""GEMM + per-head RoPE + dual-direction MXFP8 projection (oracle; test infrastructure).

"GEMM + RoPE + MXFP8 Projection (SM100)", Overview, Shapes and Equations.  MXFP8 input path:
x (tokens, K) and w (N, K) = [out, in] are E4M3 codes with E8M0 block scales along K
(block 32, plain row-major (rows, K/32) arrays), N = NUM_HEADS * HEAD_DIM; BF16 input path:
x and w are bf16 values (``project_bf16``).

    Y[t, h, :] = (xhat @ what^T)[t, h * HEAD_DIM : (h + 1) * HEAD_DIM]
    the trailing QK_ROPE features of every head are rotated (RoPE), the leading
    P = HEAD_DIM - QK_ROPE pass unchanged;
    out_row / scales_row: MXFP8 of Y in blocks of 32 consecutive features of a head;
    out_col / scales_col: MXFP8 of Y in blocks of 32 consecutive tokens of a feature.

Readings of the page taken here (each also listed in the design notes):
* "interleaved-in / halves-out" RoPE: the rotary features arrive as interleaved pairs
  (a_j, b_j) = (Y[P + 2j], Y[P + 2j + 1]), j < R/2 (R = QK_ROPE), and leave in halves:
      out[P + j]       = a_j * cos[t, j]       - b_j * sin[t, j]
      out[P + R/2 + j] = b_j * cos[t, R/2 + j] + a_j * sin[t, R/2 + j]
  which is de-interleaving into halves followed by x * cos + rotate_half(x) * sin with
  rotate_half([u, v]) = [-v, u].  cos / sin are the caller's (tokens, R) tables (YARN's
  frequency and magnitude scaling live in them); their bf16 values are used exactly.
* Y is rotated and quantised from its exact (here float64) value; the kernel does it in fp32
  from the fp32 accumulator.
* MXFP8 quantisation as for the grouped FP8 D with norm_const = 1: the block scale is the
  smallest power of two 2^e with blockamax <= 448 * 2^e, codes RNE_satfinite_E4M3(Y / 2^e).
* Scale outputs are plain row-major: scales_row (tokens, H, HEAD_DIM/32), scales_col
  (tokens/32, H, HEAD_DIM); both code outputs are (tokens, H, HEAD_DIM).

Float64 throughout; numpy's matmul is the library primitive of the GEMM.
"""
from __future__ import annotations

import numpy as np

from . import formats, gemm

BLOCK = 32


def dequantize_plain(codes, scales) -> np.ndarray:
    """E4M3 codes (R, K) with plain E8M0 scales (R, K/32) -> float64 (R, K)."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    r, k = codes.shape
    assert scales.shape == (r, k // BLOCK)
    return formats.decode_e4m3(codes) * np.repeat(formats.decode_e8m0(scales), BLOCK, axis=1)


def rope_interleaved_halves(y_rope, cos, sin) -> np.ndarray:
    """(tokens, H, R) interleaved pairs -> (tokens, H, R) rotated halves (see the header)."""
    y = np.asarray(y_rope, dtype=np.float64)
    c = np.asarray(cos, dtype=np.float64)[:, None, :]
    s = np.asarray(sin, dtype=np.float64)[:, None, :]
    half = y.shape[-1] // 2
    a, b = y[..., 0::2], y[..., 1::2]
    out = np.empty_like(y)
    out[..., :half] = a * c[..., :half] - b * s[..., :half]
    out[..., half:] = b * c[..., half:] + a * s[..., half:]
    return out


def project(x_codes, x_scales, w_codes, w_scales, cos, sin, num_heads: int, head_dim: int, qk_rope: int):
    """The MXFP8-input path.  Returns a dict: y (tokens, H, D) float64 after RoPE, out_row /
    out_col codes (tokens, H, D) uint8, scales_row (tokens, H, D/32), scales_col (tokens/32, H, D)."""
    xh = dequantize_plain(x_codes, x_scales)
    wh = dequantize_plain(w_codes, w_scales)
    return _rotate_and_quantise(xh @ wh.T, cos, sin, num_heads, head_dim, qk_rope)


def project_bf16(x_values, w_values, cos, sin, num_heads: int, head_dim: int, qk_rope: int):
    """The BF16-input path (the page's other input precision): x (tokens, K) and w (N, K) are
    the bf16 values themselves (given exactly, e.g. as float32 or float64); the rest as
    ``project``."""
    xh = np.asarray(x_values, dtype=np.float64)
    wh = np.asarray(w_values, dtype=np.float64)
    return _rotate_and_quantise(xh @ wh.T, cos, sin, num_heads, head_dim, qk_rope)


def _rotate_and_quantise(y2d, cos, sin, num_heads: int, head_dim: int, qk_rope: int):
    tokens = y2d.shape[0]
    y = np.array(y2d, dtype=np.float64).reshape(tokens, num_heads, head_dim)
    p = head_dim - qk_rope
    y[..., p:] = rope_interleaved_halves(y[..., p:], cos, sin)
    flat = y.reshape(tokens, num_heads * head_dim)
    out_row, sf_row = gemm.mxfp8_quantize_blocks(flat, 1.0, axis=1)
    out_col, sf_col = gemm.mxfp8_quantize_blocks(flat, 1.0, axis=0)
    return {"y": y,
            "out_row": out_row.reshape(tokens, num_heads, head_dim),
            "scales_row": sf_row.reshape(tokens, num_heads, head_dim // BLOCK),
            "out_col": out_col.reshape(tokens, num_heads, head_dim),
            "scales_col": sf_col.T.reshape(tokens // BLOCK, num_heads, head_dim)}

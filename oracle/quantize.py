"""Block quantiser and dequantiser (oracle; test infrastructure).

Dequantisation is the pages' definition ("GEMM + Amax (SM100)", Equations): the
value of element k of a row is decode(code) * decode(scale of block k // v), the
scales held in the scale-factor atom layout (``sf_layout``).

The quantiser produces the workloads' operands from fp32 values:

* MXFP8 (E4M3 codes, E8M0 scales, v = 32): per block of 32 values along K, the
  scale is 2^e with e the smallest integer such that blockamax <= 448 * 2^e
  (i.e. 2^ceil(log2(blockamax/448))), clamped to the E8M0 codes [0, 254]; each
  code is RNE_satfinite_E4M3(x / 2^e) on the exact quotient.
* NVFP4 (E2M1 codes, UE4M3 scales, v = 16): the scale is s = RNE_UE4M3(blockamax/6)
  and each code is RNE_satfinite_E2M1(x / s), decided exactly; s == 0 gives zero
  codes.  Two codes per byte, element 2j in the low nibble.

blockamax/6 is computed in float64: amax is an fp32 value, and it equals 6*p for
an E4M3 rounding midpoint p only when the quotient is exact, so the float64
rounding of the quotient can neither cross nor create a rounding tie.
Scale bytes of the padded extent of the atom layout are zero.
"""
from __future__ import annotations

import numpy as np

from . import formats, sf_layout

FORMATS = {
    # fmt: (sf_vec, elements per byte)
    "mxfp8": (32, 1),
    "nvfp4": (16, 2),
}


def quantize(x: np.ndarray, fmt: str):
    """Quantise fp32 ``x`` of shape (batch, rows, K) along K.

    Returns ``(codes, sf)``: codes uint8 (batch, rows, K) for MXFP8 or
    (batch, rows, K/2) packed for NVFP4; sf the flat physical scale buffer.
    """
    codes, sf = quantize_logical(x, fmt)
    return codes, sf_layout.pack(sf)


def quantize_logical(x: np.ndarray, fmt: str):
    """As ``quantize`` but returns the scale bytes in logical (batch, rows, K/v) order."""
    x = np.asarray(x, dtype=np.float32)
    if x.ndim == 2:
        x = x[None]
    batch, rows, k = x.shape
    v, _ = FORMATS[fmt]
    assert k % v == 0, "K must be a whole number of scale blocks"
    blocks = k // v
    xb = x.astype(np.float64).reshape(batch, rows, blocks, v)
    amax = np.abs(xb).max(axis=-1)
    if fmt == "mxfp8":
        sf = formats.e8m0_ceil_code(amax)
        scale = formats.decode_e8m0(sf)
        codes = formats.encode_e4m3(xb / scale[..., None]).reshape(batch, rows, k)
    else:
        sf = formats.encode_e4m3(amax / 6.0)  # non-negative: a UE4M3 code
        scale = formats.decode_ue4m3(sf)
        nib = formats.encode_e2m1_scaled(xb, scale[..., None]).reshape(batch, rows, k)
        codes = (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
    return codes, sf


def decode_codes(codes: np.ndarray, fmt: str) -> np.ndarray:
    """Element values (float64) of code bytes; NVFP4 bytes unpack to two values each."""
    codes = np.asarray(codes, dtype=np.uint8)
    if fmt == "mxfp8":
        return formats.decode_e4m3(codes)
    lo = formats.decode_e2m1(codes & 0xF)
    hi = formats.decode_e2m1(codes >> 4)
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.float64)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def decode_scales(sf_bytes: np.ndarray, fmt: str) -> np.ndarray:
    return formats.decode_e8m0(sf_bytes) if fmt == "mxfp8" else formats.decode_ue4m3(sf_bytes)


def dequantize(codes: np.ndarray, sf: np.ndarray, fmt: str, rows: int, k: int, batch: int = 1) -> np.ndarray:
    """float64 (batch, rows, K): decode(code) * decode(scale of its K block)."""
    v, _ = FORMATS[fmt]
    blocks = -(-k // v)
    vals = decode_codes(codes, fmt).reshape(batch, rows, k)
    scales = decode_scales(sf_layout.unpack(sf, rows, blocks, batch), fmt)
    return vals * np.repeat(scales, v, axis=-1)[..., :k]


def dequantize_rows(codes_rows: np.ndarray, sf: np.ndarray, fmt: str, row_ids, rows: int, k: int) -> np.ndarray:
    """Dequantise selected rows: codes_rows (len(row_ids), K or K/2), ids flat over batch*rows."""
    v, _ = FORMATS[fmt]
    blocks = -(-k // v)
    vals = decode_codes(codes_rows, fmt).reshape(len(row_ids), k)
    scales = decode_scales(sf_layout.unpack_rows(sf, row_ids, blocks, rows), fmt)
    return vals * np.repeat(scales, v, axis=-1)[..., :k]

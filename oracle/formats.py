"""Low-precision number formats used by the block-scaled GEMM (oracle; test infrastructure).

Formats named by the pages' tensor contracts ("GEMM + Amax (SM100)", Parameters:
A/B dtypes float8_e4m3fn and float4_e2m1fn_x2, scale-factor dtypes
float8_e8m0fnu and float8_e4m3fn):

* E4M3 (float8_e4m3fn): 1 sign, 4 exponent (bias 7), 3 mantissa bits, subnormals,
  no infinities, 0x7F/0xFF are NaN, largest finite 448.
* E2M1 (one nibble of float4_e2m1fn_x2): 1 sign, 2 exponent (bias 1), 1 mantissa
  bit: magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
* E8M0 (float8_e8m0fnu): an unsigned power of two 2^(code-127); 0xFF is NaN.
* UE4M3: the E4M3 value grid used as an (unsigned) NVFP4 block scale.

Decoders are the formulas above.  Encoders round to nearest, ties to the even
code, saturating to the largest finite magnitude ("satfinite"); the decision is
taken on the exact input value, so a float64 input that is itself exact gives
the correctly rounded code.  As in IEEE rounding the sign is kept, so a negative
value that rounds to zero encodes as -0.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E2M1_MAX = 6.0
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
# midpoints between consecutive E2M1 magnitudes
E2M1_MIDS = (E2M1_GRID[:-1] + E2M1_GRID[1:]) / 2.0


def decode_e4m3(codes) -> np.ndarray:
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & ((c & 7) == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def decode_ue4m3(codes) -> np.ndarray:
    """Unsigned E4M3 scale: the E4M3 magnitude of bits 0-6 (bit 7 is never set by the quantiser)."""
    return decode_e4m3(np.asarray(codes).astype(np.int64) & 0x7F)


def decode_e2m1(nibbles) -> np.ndarray:
    n = np.asarray(nibbles).astype(np.int64) & 0xF
    sign = (n >> 3) & 1
    e = (n >> 1) & 3
    m = (n & 1).astype(np.float64)
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e.astype(np.float64) - 1.0))
    return np.where(sign == 1, -mag, mag)


def decode_e8m0(codes) -> np.ndarray:
    c = np.asarray(codes).astype(np.int64) & 0xFF
    return np.where(c == 255, np.nan, np.exp2(c.astype(np.float64) - 127.0))


def encode_e4m3(x) -> np.ndarray:
    """RNE + satfinite E4M3 code of each (exact) float64 value; NaN inputs are not expected."""
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.minimum(np.abs(x), E4M3_MAX)
    # subnormal range: multiples of 2^-9 below 2^-6 (the count 8 is code 0x08 = 2^-6)
    q_sub = np.rint(a * 2.0 ** 9)  # exact scaling; rint rounds half to even
    # normal range: a = (1 + f/8) * 2^E, so a * 2^(3-E) lies in [8, 16)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    big_e = ex.astype(np.int64) - 1
    q = np.rint(a * np.exp2((3 - big_e).astype(np.float64)))
    carry = q >= 16
    big_e = np.where(carry, big_e + 1, big_e)
    q = np.where(carry, 8, q)
    code_norm = ((big_e + 7) << 3) | (q.astype(np.int64) - 8)
    code = np.where(a < 2.0 ** -6, q_sub.astype(np.int64), code_norm)
    # rounding keeps the sign: a negative value that rounds to zero gives -0 (0x80)
    code = np.where(neg, code | 0x80, code)
    return code.astype(np.uint8)


def encode_e2m1_scaled(x, s) -> np.ndarray:
    """E2M1 nibble of RNE_satfinite(x / s) decided exactly: |x| is compared with midpoint*s.

    ``x`` and ``s`` are float64 arrays (broadcastable); every midpoint has at most
    three significant bits and ``s`` at most four, so ``midpoint*s`` is exact and
    no quotient is ever rounded.  ``s == 0`` gives code 0.
    """
    x = np.asarray(x, dtype=np.float64)
    s = np.asarray(s, dtype=np.float64)
    a = np.abs(x)
    idx = np.zeros(np.broadcast(a, s).shape, dtype=np.int64)
    for i, mid in enumerate(E2M1_MIDS):
        thr = mid * s
        above = a > thr
        tie = a == thr
        # on a tie the even of (i, i+1) wins
        even_up = (i + 1) % 2 == 0
        idx = idx + np.where(above | (tie & even_up), 1, 0)
    # rounding keeps the sign (a negative value that rounds to zero gives -0, nibble 0x8);
    # a zero scale gives the code +0 for every element
    neg = np.signbit(x) & (s > 0)
    idx = np.where(s > 0, idx, 0)
    return (idx | np.where(neg, 8, 0)).astype(np.uint8)


def e8m0_ceil_code(amax, limit: float = E4M3_MAX) -> np.ndarray:
    """E8M0 code of the smallest power of two 2^e with amax <= limit * 2^e, clamped to [0, 254].

    amax = f * 2^x with f in [0.5, 1) (frexp, exact); limit = 448 = 0.875 * 2^9, so
    the condition is e = x - 9 when f <= 0.875 and e = x - 8 otherwise.  A zero
    block clamps to code 0.
    """
    amax = np.asarray(amax, dtype=np.float64)
    lf, lx = np.frexp(limit)
    f, x = np.frexp(np.where(amax > 0, amax, 1.0))
    e = np.where(f <= lf, x - lx, x - lx + 1).astype(np.int64)
    code = np.where(amax > 0, e + 127, 0)
    return np.clip(code, 0, 254).astype(np.uint8)


def bf16_round(x) -> np.ndarray:
    """Round float64 values to bfloat16 (8 significant bits, RNE) and return them as float64.

    x = f * 2^e with f in [0.5, 1), so x * 2^(8-e) lies in [128, 256); rounding that
    (exact) value to an integer, ties to even, and scaling back gives the bfloat16
    value.  Normal range only (the workloads never reach bfloat16 subnormals).
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(np.where(x != 0, x, 1.0))
    e = e.astype(np.float64)
    return np.where(x != 0, np.rint(x * np.exp2(8.0 - e)) * np.exp2(e - 8.0), 0.0)


def bf16_ulp(x) -> np.ndarray:
    """Spacing of bfloat16 numbers at |x| (8 significant bits; subnormals ignored)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    _, ex = np.frexp(np.where(a > 0, a, 2.0 ** -126))
    return np.exp2(ex.astype(np.float64) - 8.0)


def f16_round(x) -> np.ndarray:
    """Round float64 values to IEEE half precision (RNE, saturating to +-inf beyond 65504 as
    the conversion does) and return them as float64; numpy's conversion is the library step."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def f16_ulp(x) -> np.ndarray:
    """Spacing of half-precision numbers at |x| (11 significant bits; 2^-24 in the subnormal range)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    _, ex = np.frexp(np.where(a > 0, a, 2.0 ** -14))
    return np.maximum(np.exp2(ex.astype(np.float64) - 11.0), 2.0 ** -24)


def encode_e2m1(x) -> np.ndarray:
    """E2M1 nibble of RNE_satfinite(x) for float64 x (a plain conversion, scale 1)."""
    return encode_e2m1_scaled(x, 1.0)


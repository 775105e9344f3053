"""Tolerance checks shared by the GPU parity tests.

The acceptance rules (derived from the arithmetic; the reasoning is in the design notes):

* scale-factor bytes, codes of the input quantiser, offsets handling: bit-exact;
* fp32 C:  |C - ref| <= 2^-20 * alpha * sum_k |Ahat||Bhat|   (the stated accumulation bound);
* bf16 C:  the same plus one bf16 ulp of ref (the final rounding);
* amax:    relative error <= 1e-5;
* bf16 D:  |D - ref| <= 1 bf16 ulp(ref) + prob * 2|C_ref| * tolC + 2^-20 |ref|, i.e. the
           one-ulp rule plus the C tolerance carried through d(r^2) = 2r dr (the clamp's
           derivative is smaller) and fp32 epilogue rounding;
* dSwiGLU D (ab, dswiglu): the ref bound carried through the (linear in ref) epilogue, plus
           the fp32 epilogue: a relative 2^-20 (1 + |gate|) for the fast exponential (its error
           grows with the argument) and division, applied to each factor so the cancellation in
           1 + gate (1 - sigmoid) is covered; then one ulp of the output type;
* dprob:   the carried ref bound plus fp32 summation over the kernel's partial sums;
* E4M3 D / D_col: codes equal, except a neighbouring code where the oracle's pre-quantised
           value lies within max(1e-5 relative, carried C tolerance) of the rounding boundary;
           a block scale may differ by one code where the oracle's block amax lies that close to
           a power-of-two boundary of 448 * 2^e, and that block is then checked by value.
"""
from __future__ import annotations

import numpy as np

from oracle import formats

TOL_C = 2.0 ** -20


def check_c(c_gpu, ref, abs_sum, kind: str, scale=1.0, what="C"):
    c_gpu = np.asarray(c_gpu, dtype=np.float64)
    tol = TOL_C * np.abs(scale) * abs_sum
    if kind == "bf16":
        tol = tol + formats.bf16_ulp(ref)
    err = np.abs(c_gpu - ref)
    bad = ~(err <= tol)
    if bad.any():
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first "
                             f"gpu={c_gpu.ravel()[i]} ref={ref.ravel()[i]} tol={np.broadcast_to(tol, ref.shape).ravel()[i]}")


def check_c_float(c_gpu, ref, abs_sum, kind: str, scale=1.0, what="C"):
    """fp32 / bf16 / f16 C: the accumulation bound plus one unit in the last place of the output."""
    c_gpu = np.asarray(c_gpu, dtype=np.float64)
    tol = TOL_C * np.abs(scale) * abs_sum
    if kind == "bf16":
        tol = tol + formats.bf16_ulp(ref)
    elif kind == "f16":
        tol = tol + formats.f16_ulp(ref)
    err = np.abs(c_gpu - ref)
    bad = ~(err <= tol)
    if bad.any():
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first "
                             f"gpu={c_gpu.ravel()[i]} ref={ref.ravel()[i]} tol={np.broadcast_to(tol, ref.shape).ravel()[i]}")


def _e2m1_rank(nib):
    n = np.asarray(nib).astype(np.int64)
    return np.where(n & 8, -(n & 7), n & 7)


def check_codes_plain(codes_gpu, ref, tol, kind: str, what="C"):
    """Plain (unscaled) E4M3 / E2M1 conversions of C: codes equal to the oracle's RNE_satfinite
    of the exact value, except a neighbouring code where the exact value lies within `tol` of
    the rounding midpoint between the two."""
    ref = np.asarray(ref, dtype=np.float64)
    if kind == "e4m3":
        want = formats.encode_e4m3(ref)
        got = np.asarray(codes_gpu, dtype=np.uint8)
        rank_g, rank_w = _rank(got), _rank(want)
        dec = formats.decode_e4m3
    else:
        want = formats.encode_e2m1(ref)
        g = np.asarray(codes_gpu, dtype=np.uint8)
        got = np.empty(g.shape[:-1] + (g.shape[-1] * 2,), dtype=np.uint8)
        got[..., 0::2] = g & 0xF
        got[..., 1::2] = g >> 4
        rank_g, rank_w = _e2m1_rank(got), _e2m1_rank(want)
        dec = formats.decode_e2m1
    # +0 and -0 are the same value (the sign of a tiny C may differ within the C bound)
    mism = (want != got) & ~((dec(want) == 0) & (dec(got) == 0))
    if mism.any():
        vg, vw = dec(got[mism]), dec(want[mism])
        adjacent = np.abs(rank_g[mism] - rank_w[mism]) == 1
        near = np.abs(ref[mism] - (vg + vw) / 2.0) <= np.broadcast_to(tol, ref.shape)[mism] + 1e-12
        if not np.all(adjacent & near):
            k = np.flatnonzero(~(adjacent & near))[:5]
            raise AssertionError(f"{what}: {(~(adjacent & near)).sum()} codes differ away from a rounding "
                                 f"midpoint; ref={ref[mism][k]} gpu={vg[k]} want={vw[k]}")


def check_amax(amax_gpu, ref, what="amax"):
    amax_gpu = np.asarray(amax_gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(amax_gpu - ref)
    ok = err <= 1e-5 * np.abs(ref)
    if not np.all(ok):
        raise AssertionError(f"{what}: gpu={amax_gpu[~ok][:5]} ref={ref[~ok][:5]}")


def d_tolerance(c_ref, prob, c_tol):
    """Absolute error of fp32 D carried from the C error bound."""
    return np.asarray(prob, np.float64).reshape(-1, 1) * 2.0 * np.maximum(c_ref, 0.0) * c_tol


def check_d_bf16(d_gpu, d_ref, c_ref, prob, c_tol, what="D"):
    d_gpu = np.asarray(d_gpu, dtype=np.float64)
    tol = formats.bf16_ulp(d_ref) + d_tolerance(c_ref, prob, c_tol) + 2.0 ** -20 * np.abs(d_ref)
    err = np.abs(d_gpu - d_ref)
    bad = ~(err <= tol)
    if bad.any():
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first gpu={d_gpu.ravel()[i]} "
                             f"ref={d_ref.ravel()[i]} tol={tol.ravel()[i]}")


def check_d_float(d_gpu, d_ref, c_ref, prob, c_tol, kind: str, what="D"):
    """bf16 / f16 / f32 D: one unit in the last place of the output type (none for f32) plus
    the C bound carried through d(r^2) = 2r dr and fp32 epilogue rounding."""
    if kind == "bf16":
        return check_d_bf16(d_gpu, d_ref, c_ref, prob, c_tol, what)
    d_gpu = np.asarray(d_gpu, dtype=np.float64)
    ulp = formats.f16_ulp(d_ref) if kind == "f16" else 0.0
    tol = ulp + d_tolerance(c_ref, prob, c_tol) + 2.0 ** -20 * np.abs(d_ref)
    err = np.abs(d_gpu - d_ref)
    bad = ~(err <= tol)
    if bad.any():
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first gpu={d_gpu.ravel()[i]} "
                             f"ref={d_ref.ravel()[i]} tol={np.broadcast_to(tol, d_ref.shape).ravel()[i]}")


def _rank(codes):
    """Position of E4M3 codes in value order (sign-magnitude -> signed integer)."""
    c = np.asarray(codes).astype(np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def check_e4m3_blocks(codes_gpu, sf_gpu, d_ref, d_tol, nc: float, axis: int, what="D"):
    """Checks E4M3 codes + E8M0 block scales of D quantised in blocks of 32 along ``axis``.

    codes_gpu (R, C) uint8; sf_gpu logical scale codes (R, C/32) for axis 1 or (C, R/32)
    for axis 0; d_ref / d_tol float64 (R, C).  Returns (number of scale codes that differ,
    number of element codes that differ) for reporting.
    """
    x = d_ref if axis == 1 else d_ref.T
    t = d_tol if axis == 1 else d_tol.T
    q = np.asarray(codes_gpu if axis == 1 else codes_gpu.T)
    r, c = x.shape
    xb, tb, qb = x.reshape(r, c // 32, 32), t.reshape(r, c // 32, 32), q.reshape(r, c // 32, 32)
    sf_gpu = np.asarray(sf_gpu).astype(np.int64)
    amax = np.abs(xb).max(-1)
    sf_ref = formats.e8m0_ceil_code(nc * amax).astype(np.int64)
    # block-scale mismatches: only next to a 448 * 2^e boundary, and by one code
    diff_sf = sf_gpu != sf_ref
    if diff_sf.any():
        e = np.minimum(sf_gpu, sf_ref)[diff_sf] - 127
        boundary = 448.0 * np.exp2(e.astype(np.float64))
        amax_tol = nc * np.take_along_axis(tb, np.abs(xb).argmax(-1)[..., None], -1)[..., 0][diff_sf]
        near = np.abs(nc * amax[diff_sf] - boundary) <= np.maximum(1e-5 * boundary, amax_tol)
        if not (np.all(np.abs(sf_gpu[diff_sf] - sf_ref[diff_sf]) == 1) and np.all(near)):
            raise AssertionError(f"{what}: {diff_sf.sum()} block scales differ away from a boundary")
    same = ~diff_sf
    scale = formats.decode_e8m0(sf_ref)[..., None]
    v = xb * nc / scale  # the oracle's pre-quantised values
    want = formats.encode_e4m3(v)
    got = qb
    mism = (want != got) & same[..., None]
    if mism.any():
        vg = formats.decode_e4m3(got[mism])
        vw = formats.decode_e4m3(want[mism])
        adjacent = np.abs(_rank(got[mism]) - _rank(want[mism])) == 1
        boundary = (vg + vw) / 2.0
        delta = np.maximum(1e-5 * np.abs(v[mism]), (tb * nc / scale)[mism])
        near = np.abs(v[mism] - boundary) <= delta
        if not np.all(adjacent & near):
            k = np.flatnonzero(~(adjacent & near))[:5]
            raise AssertionError(f"{what}: {(~(adjacent & near)).sum()} codes differ away from a rounding "
                                 f"boundary; v={v[mism][k]} gpu={vg[k]} want={vw[k]}")
    # blocks whose scale differs: compare dequantised values with D
    if diff_sf.any():
        sg = formats.decode_e8m0(sf_gpu)[..., None]
        deq = formats.decode_e4m3(qb) * sg / nc
        err = np.abs(deq - xb)[diff_sf]
        bound = (np.maximum(np.abs(xb) * 2.0 ** -4, 2.0 ** -10 * sg / nc) + tb)[diff_sf]
        if not np.all(err <= bound * (1 + 1e-9)):
            raise AssertionError(f"{what}: values of re-scaled blocks outside half an E4M3 ulp")
    return int(diff_sf.sum()), int(mism.sum())


def dswiglu_tolerances(ref_out, ref_tol, prob):
    """Absolute bounds (float64, (valid_m, N) each) on the fp32 ab and dswiglu values, from the
    oracle's exact x, gate and ref and the ref bound ``ref_tol``."""
    p = np.asarray(prob, np.float64).reshape(-1, 1)
    x, g, ref = ref_out["x"], ref_out["gate"], ref_out["ref"]
    sig = 1.0 / (1.0 + np.exp(-np.clip(g, -700, 700)))
    sw = g * sig
    h = 1.0 + g * (1.0 - sig)
    eps = 2.0 ** -20 * (1.0 + np.abs(g))
    tol_ab = p * np.abs(sw) * ref_tol + eps * np.abs(ref_out["ab"]) + 1e-30
    base = np.abs(ref * p * x * sig)
    tol_dsw = p * np.abs(x * sig * h) * ref_tol + base * eps * (1.0 + np.abs(h) + np.abs(g)) + 1e-30
    return tol_ab, tol_dsw


def check_float_out(got, ref, tol, kind: str, what="D"):
    """bf16 / f16 / f32 output: |got - ref| <= one ulp of the output type (none for f32) + tol."""
    got = np.asarray(got, dtype=np.float64)
    ulp = formats.bf16_ulp(ref) if kind == "bf16" else formats.f16_ulp(ref) if kind == "f16" else 0.0
    err = np.abs(got - ref)
    bad = ~(err <= ulp + tol)
    if bad.any():
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first gpu={got.ravel()[i]} "
                             f"ref={np.asarray(ref).ravel()[i]} tol={np.broadcast_to(tol, np.shape(ref)).ravel()[i]}")


def dprob_tolerance(ref_out, ref_tol, terms_per_partial: int, partials: int):
    """Bound on the fp32 dprob: the carried ref bound, the epilogue's relative error and the
    rounding of a sum of ``terms_per_partial`` terms per partial and ``partials`` partial sums
    added in any order."""
    x, g, ref = ref_out["x"], ref_out["gate"], ref_out["ref"]
    sig = 1.0 / (1.0 + np.exp(-np.clip(g, -700, 700)))
    sw = g * sig
    terms = np.abs(sw * x * ref)
    eps = 2.0 ** -20 * (1.0 + np.abs(g))
    depth = terms_per_partial + partials + 4
    return (np.sum(np.abs(sw * x) * ref_tol, axis=1) + np.sum(eps * terms, axis=1) +
            depth * 2.0 ** -23 * np.sum(terms, axis=1) + 1e-30)

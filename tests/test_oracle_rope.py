"""Pins of the GEMM + RoPE + MXFP8 projection oracle ("GEMM + RoPE + MXFP8 Projection (SM100)").

* the rotation against complex multiplication (a + i b) e^{i theta} on de-interleaved pairs;
* special angles (identity = de-interleave; a quarter turn) and norm preservation;
* the leading no-position features and the whole path against scalar loops on a tiny case;
* plain scale layouts: every block's scale covers its amax and is the smallest that does.
"""
import math

import numpy as np
import pytest

from oracle import formats, quantize, rope


def _tables(tokens, r, rng, mscale=1.0):
    theta = rng.uniform(0, 2 * math.pi, size=(tokens, r // 2))
    th = np.concatenate([theta, theta], axis=1)  # the same angle for both halves of a pair
    return mscale * np.cos(th), mscale * np.sin(th), theta


def test_rotation_is_complex_multiplication():
    rng = np.random.default_rng(0)
    tokens, h, r = 5, 3, 64
    y = rng.standard_normal((tokens, h, r))
    cos, sin, theta = _tables(tokens, r, rng)
    out = rope.rope_interleaved_halves(y, cos, sin)
    z = (y[..., 0::2] + 1j * y[..., 1::2]) * np.exp(1j * theta)[:, None, :]
    np.testing.assert_allclose(out[..., :r // 2], z.real, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(out[..., r // 2:], z.imag, rtol=1e-13, atol=1e-13)
    # norm of every pair preserved
    n_in = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    n_out = out[..., :r // 2] ** 2 + out[..., r // 2:] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12)


def test_special_angles():
    rng = np.random.default_rng(1)
    y = rng.standard_normal((2, 1, 8))
    ident = rope.rope_interleaved_halves(y, np.ones((2, 8)), np.zeros((2, 8)))
    for j in range(4):
        assert np.array_equal(ident[..., j], y[..., 2 * j])
        assert np.array_equal(ident[..., 4 + j], y[..., 2 * j + 1])
    quarter = rope.rope_interleaved_halves(y, np.zeros((2, 8)), np.ones((2, 8)))
    np.testing.assert_array_equal(quarter[..., :4], -y[..., 1::2])
    np.testing.assert_array_equal(quarter[..., 4:], y[..., 0::2])
    # per-half tables: the second half may carry its own cos / sin
    c = np.concatenate([np.full((2, 4), 0.5), np.full((2, 4), 2.0)], axis=1)
    s = np.concatenate([np.full((2, 4), 3.0), np.full((2, 4), -1.0)], axis=1)
    o = rope.rope_interleaved_halves(y, c, s)
    np.testing.assert_allclose(o[..., 1], 0.5 * y[..., 2] - 3.0 * y[..., 3])
    np.testing.assert_allclose(o[..., 5], 2.0 * y[..., 3] - 1.0 * y[..., 2])


def test_whole_path_scalar_loops():
    rng = np.random.default_rng(2)
    tokens, k, h, d, r = 64, 64, 2, 96, 64
    x = rng.standard_normal((1, tokens, k)).astype(np.float32)
    w = (rng.standard_normal((1, h * d, k)) / 8).astype(np.float32)
    xc, xs = quantize.quantize_logical(x, "mxfp8")
    wc, ws = quantize.quantize_logical(w, "mxfp8")
    cos, sin, _ = _tables(tokens, r, rng, mscale=1.2)
    out = rope.project(xc[0], xs[0], wc[0], ws[0], cos, sin, h, d, r)
    xh = formats.decode_e4m3(xc[0]) * np.repeat(formats.decode_e8m0(xs[0]), 32, axis=1)
    wh = formats.decode_e4m3(wc[0]) * np.repeat(formats.decode_e8m0(ws[0]), 32, axis=1)

    def yraw(t, head, f):
        return sum(float(xh[t, kk]) * float(wh[head * d + f, kk]) for kk in range(k))

    p = d - r
    for t, head, f in [(0, 0, 0), (5, 1, p - 1), (63, 0, 17)]:
        assert out["y"][t, head, f] == pytest.approx(yraw(t, head, f), rel=1e-12, abs=1e-12)
    for t, head, j in [(0, 0, 0), (9, 1, 31), (40, 0, 13)]:
        a, b = yraw(t, head, p + 2 * j), yraw(t, head, p + 2 * j + 1)
        assert out["y"][t, head, p + j] == pytest.approx(a * cos[t, j] - b * sin[t, j], rel=1e-11, abs=1e-12)
        assert out["y"][t, head, p + 32 + j] == pytest.approx(b * cos[t, 32 + j] + a * sin[t, 32 + j], rel=1e-11,
                                                              abs=1e-12)


def test_scale_layouts_cover_blocks():
    rng = np.random.default_rng(3)
    tokens, k, h, d, r = 64, 32, 3, 64, 32
    xc, xs = quantize.quantize_logical(rng.standard_normal((1, tokens, k)).astype(np.float32), "mxfp8")
    wc, ws = quantize.quantize_logical(rng.standard_normal((1, h * d, k)).astype(np.float32), "mxfp8")
    cos, sin, _ = _tables(tokens, r, rng)
    out = rope.project(xc[0], xs[0], wc[0], ws[0], cos, sin, h, d, r)
    y = out["y"]
    assert out["scales_row"].shape == (tokens, h, d // 32) and out["scales_col"].shape == (tokens // 32, h, d)
    amax_row = np.abs(y.reshape(tokens, h, d // 32, 32)).max(-1)
    amax_col = np.abs(y.reshape(tokens // 32, 32, h, d)).max(1)
    for amax, sf in ((amax_row, out["scales_row"]), (amax_col, out["scales_col"])):
        scale = formats.decode_e8m0(sf)
        assert np.all(amax <= 448 * scale)
        nz = amax > 0
        assert np.all(amax[nz] > 448 * scale[nz] / 2)  # the smallest such power of two
    # dequantised row codes are within half an E4M3 step of Y
    deq = formats.decode_e4m3(out["out_row"]) * np.repeat(formats.decode_e8m0(out["scales_row"]), 32, axis=-1)
    assert np.all(np.abs(deq - y) <= np.abs(y) * 2.0 ** -4 + 2.0 ** -10 * np.repeat(
        formats.decode_e8m0(out["scales_row"]), 32, axis=-1))


def test_bf16_path_matches_the_mxfp8_path_on_shared_values():
    """Inputs whose MXFP8 encoding is exact are also bf16 values: both input paths must give the
    same projection and outputs."""
    rng = np.random.default_rng(5)
    tokens, k, h, d, r = 64, 64, 2, 96, 64
    grid = formats.decode_e4m3(np.arange(0, 0x7F, dtype=np.uint8))
    grid = grid[(grid >= 0.125) & (grid <= 8)]
    x = (rng.choice(grid, (tokens, k)) * rng.choice([-1, 1], (tokens, k))).astype(np.float32)
    w = (rng.choice(grid, (h * d, k)) * rng.choice([-1, 1], (h * d, k)) / 16).astype(np.float32)
    # each block's amax (8 and 0.5) fixes its scale (2^-5, 2^-9), under which every value is an
    # exact E4M3 code
    x[:, ::32] = 8.0
    w[:, ::32] = 0.5
    xc, xs = quantize.quantize_logical(x[None], "mxfp8")
    wc, wsc = quantize.quantize_logical(w[None], "mxfp8")
    np.testing.assert_array_equal(rope.dequantize_plain(xc[0], xs[0]), x)
    np.testing.assert_array_equal(rope.dequantize_plain(wc[0], wsc[0]), w)
    cos, sin, _ = _tables(tokens, r, rng)
    a = rope.project(xc[0], xs[0], wc[0], wsc[0], cos, sin, h, d, r)
    b = rope.project_bf16(x, w, cos, sin, h, d, r)
    for key in ("y", "out_row", "scales_row", "out_col", "scales_col"):
        np.testing.assert_array_equal(a[key], b[key])

"""Pins of the oracle's number formats against library decoders, the formats' tables and brute force."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import formats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_decode(codes, dtype):
    return torch.tensor(np.asarray(codes, np.uint8)).view(dtype).to(torch.float64).numpy()


def test_e4m3_decode_matches_torch_all_codes():
    c = np.arange(256)
    ours = formats.decode_e4m3(c)
    ref = _torch_decode(c, torch.float8_e4m3fn)
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.all((ours == ref) | both_nan)
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x38] == 1.0


def test_e8m0_decode_matches_torch_all_codes():
    c = np.arange(256)
    ours = formats.decode_e8m0(c)
    ref = _torch_decode(c, torch.float8_e8m0fnu)
    assert np.all((ours == ref) | (np.isnan(ours) & np.isnan(ref)))


def test_e2m1_decode_table():
    # the E2M1 value table: magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6 and their negatives
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    ours = formats.decode_e2m1(np.arange(16))
    assert list(ours[:8]) == table
    assert list(-ours[8:]) == table


def test_e4m3_encode_roundtrip_all_finite_codes():
    c = np.arange(256)
    v = formats.decode_e4m3(c)
    fin = ~np.isnan(v)
    assert np.array_equal(formats.encode_e4m3(v[fin]), c[fin].astype(np.uint8))  # -0.0 -> 0x80


def test_e4m3_encode_midpoints_go_to_even():
    pos = formats.decode_e4m3(np.arange(0, 0x7F))  # 0 .. 448, increasing
    mids = (pos[:-1] + pos[1:]) / 2
    got = formats.encode_e4m3(mids).astype(np.int64)
    lo = np.arange(0, 0x7E)
    want = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(got, want)
    # just off the midpoint goes to the nearer neighbour
    eps = (pos[1:] - pos[:-1]) * 1e-6
    assert np.array_equal(formats.encode_e4m3(mids - eps), lo.astype(np.uint8))
    assert np.array_equal(formats.encode_e4m3(mids + eps), (lo + 1).astype(np.uint8))


def test_e4m3_encode_matches_torch_in_range_and_saturates():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-12, 9, 200000))).astype(np.float32)
    x = x[np.abs(x) <= 448]
    x = np.concatenate([x, np.float32([-1e-9, -2.0 ** -10, -0.0, 1e-9])])  # negatives that round to -0
    ref = torch.tensor(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = formats.encode_e4m3(x.astype(np.float64))
    assert np.array_equal(ours, ref)
    assert ours[-4:].tolist() == [0x80, 0x80, 0x80, 0x00]
    assert formats.encode_e4m3(np.array([1e9, -1e9, 460.0, 470.0])).tolist() == [0x7E, 0xFE, 0x7E, 0x7E]


def _e2m1_nearest_bruteforce(q):
    """Nearest E2M1 magnitude index by distance, ties to the even index (independent method)."""
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    out = []
    for v in np.abs(q):
        d = np.abs(grid - min(v, 6.0))
        best = np.flatnonzero(d == d.min())
        out.append(best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0])
    return np.array(out)


def test_e2m1_encode_exact_vs_bruteforce():
    rng = np.random.default_rng(2)
    s_codes = rng.integers(1, 0x7F, 4000)
    s = formats.decode_ue4m3(s_codes)
    # values at random, plus exact grid points and exact midpoints times s
    grid_pts = np.concatenate([formats.E2M1_GRID, formats.E2M1_MIDS, [7.0, 100.0]])
    q = np.concatenate([rng.uniform(-8, 8, 4000), rng.choice(grid_pts, 4000) * rng.choice([-1, 1], 4000)])
    s_all = np.concatenate([s, s])
    x = q * s_all  # exact (few significant bits)
    got = formats.encode_e2m1_scaled(x, s_all)
    want_idx = _e2m1_nearest_bruteforce(x / s_all)
    assert np.array_equal(got & 7, want_idx)
    assert np.all((got >> 3) == np.signbit(x))  # the sign is kept, -0 included
    assert np.all(formats.encode_e2m1_scaled(np.array([1.0, -3.0]), np.array([0.0, 0.0])) == 0)


def test_e8m0_ceil_code_bruteforce():
    rng = np.random.default_rng(3)
    amax = np.abs(rng.standard_normal(5000)) * np.exp2(rng.integers(-60, 60, 5000))
    amax = np.concatenate([amax, 448.0 * np.exp2(np.arange(-20, 20)), 448.0 * np.exp2(np.arange(-20, 20)) * (1 + 2**-40)])
    code = formats.e8m0_ceil_code(amax).astype(np.int64)
    e = code - 127
    assert np.all(amax <= 448.0 * np.exp2(e.astype(float)))
    assert np.all(amax > 448.0 * np.exp2(e.astype(float) - 1))
    assert formats.e8m0_ceil_code(np.array([0.0]))[0] == 0
    assert formats.e8m0_ceil_code(np.array([1e-45]))[0] == 0  # clamps at 2^-127


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(4)
    x = rng.standard_normal(100000) * np.exp2(rng.integers(-30, 30, 100000))
    ref = torch.tensor(x).to(torch.bfloat16).to(torch.float64).numpy()
    # torch rounds f64 -> bf16 directly (single rounding), which is what we compare against
    assert np.array_equal(formats.bf16_round(x), ref)


def test_f16_round_and_ulp():
    # values fixed by the binary16 format: 11 significant bits, ties to even, max 65504
    x = np.array([1.0, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 2049.0, 2051.0, 65504.0, 2.0 ** -24, 2.0 ** -26])
    want = np.array([1.0, 1.0, 1.0 + 2.0 ** -9, 2048.0, 2052.0, 65504.0, 2.0 ** -24, 0.0])
    assert np.array_equal(formats.f16_round(x), want)
    assert np.array_equal(formats.f16_ulp(np.array([1.0, 1.5, 2.0, 2.0 ** -20])),
                          np.array([2.0 ** -10, 2.0 ** -10, 2.0 ** -9, 2.0 ** -24]))


def test_e2m1_plain_conversion():
    # the E2M1 grid and its midpoints: ties go to the even code, beyond 6 saturates
    x = np.array([0.2, 0.25, 0.3, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 5.1, 100.0, -0.75, -0.1])
    mag = np.array([0, 0, 1, 2, 2, 4, 4, 6, 6, 7, 7, 2, 0])
    got = formats.encode_e2m1(x)
    assert np.array_equal(got & 7, mag)
    assert np.array_equal(got >> 3, (x < 0).astype(np.uint8))


def test_golden_worked_block_mxfp8():
    from oracle import quantize
    g = json.load(open(os.path.join(GOLDEN, "mxfp8_block_worked.json")))
    x = np.array(g["x"], dtype=np.float32).reshape(1, 1, 32)
    codes, sf = quantize.quantize_logical(x, "mxfp8")
    assert int(sf[0, 0, 0]) == g["scale_code"]
    assert codes.ravel().tolist() == g["codes"]


def test_golden_worked_block_nvfp4():
    from oracle import quantize
    g = json.load(open(os.path.join(GOLDEN, "nvfp4_block_worked.json")))
    x = np.array(g["x"], dtype=np.float32).reshape(1, 1, 32)
    codes, sf = quantize.quantize_logical(x, "nvfp4")
    assert sf.ravel().tolist() == g["scale_codes"]
    assert codes.ravel().tolist() == g["packed"]


@pytest.mark.parametrize("planted", ["drop_subnormal", "round_half_up"])
def test_planted_mistakes_are_caught(planted):
    """A plausible mistake planted in a copy of the encoder is caught by the pins above."""
    c = np.arange(0, 0x7F)
    pos = formats.decode_e4m3(c)
    mids = (pos[:-1] + pos[1:]) / 2
    if planted == "drop_subnormal":
        bad = np.where(pos < 2.0 ** -6, 0, formats.encode_e4m3(pos))
        assert not np.array_equal(bad, c.astype(np.uint8))
    else:
        bad = formats.encode_e4m3(mids * (1 + 1e-12))
        lo = np.arange(0, 0x7E)
        want = np.where(lo % 2 == 0, lo, lo + 1)
        assert not np.array_equal(bad, want)

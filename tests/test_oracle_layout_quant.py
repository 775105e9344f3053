"""Pins of the scale-factor layout and of the input quantiser."""
import json
import os

import numpy as np
import torch

from oracle import formats, quantize, sf_layout

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_offset_golden_cases():
    g = json.load(open(os.path.join(GOLDEN, "sf_layout_offsets.json")))
    for r, kb, l, off in g["cases"]:
        assert int(sf_layout.offset(r, kb, l, g["rows"], g["blocks"])) == off


def test_offset_is_bijection_over_padded_extent():
    rows, blocks, batch = 384, 12, 2
    l, r, kb = np.meshgrid(np.arange(batch), np.arange(rows), np.arange(blocks), indexing="ij")
    off = sf_layout.offset(r, kb, l, rows, blocks).ravel()
    assert len(np.unique(off)) == off.size == sf_layout.nbytes(rows, blocks, batch)


def test_pack_matches_torch_permuted_physical_view():
    """The physical (L, MT, KT, 32, 4, 4) buffer permuted by (3,4,1,5,2,0) is the logical view."""
    rows, blocks, batch = 256 + 40, 4 * 3 + 2, 2  # ragged rows and blocks
    rng = np.random.default_rng(0)
    logical = rng.integers(1, 255, (batch, rows, blocks)).astype(np.uint8)
    phys = torch.zeros(sf_layout.physical_shape(rows, blocks, batch), dtype=torch.uint8)
    view = phys.permute(3, 4, 1, 5, 2, 0)  # (32, 4, MT, 4, KT, L)
    for l in range(batch):
        for r in range(rows):
            for kb in range(blocks):
                view[r % 32, (r % 128) // 32, r // 128, kb % 4, kb // 4, l] = int(logical[l, r, kb])
    assert np.array_equal(sf_layout.pack(logical), phys.numpy().ravel())
    assert np.array_equal(sf_layout.unpack(sf_layout.pack(logical), rows, blocks, batch), logical)


def test_pack_padding_is_zero():
    logical = np.full((1, 130, 5), 0x7F, np.uint8)
    buf = sf_layout.pack(logical)
    assert buf.size == sf_layout.nbytes(130, 5) == 2 * 2 * 512
    assert (buf == 0x7F).sum() == 130 * 5 and (buf == 0).sum() == buf.size - 130 * 5


def test_mxfp8_quantiser_invariants():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((2, 64, 256)) * np.exp2(rng.integers(-20, 20, (2, 64, 1)))).astype(np.float32)
    x[0, 3, 32:64] = 0  # an all-zero block
    codes, sf = quantize.quantize_logical(x, "mxfp8")
    vals = formats.decode_e4m3(codes).reshape(2, 64, 8, 32)
    scale = formats.decode_e8m0(sf)
    bmax = np.abs(vals).max(-1)
    nz = np.abs(x.reshape(2, 64, 8, 32)).max(-1) > 0
    assert np.all((bmax[nz] >= 224) & (bmax[nz] <= 448))   # ceil recipe keeps the top binade used
    assert sf[0, 3, 1] == 0 and np.all(codes[0, 3, 32:64] == 0)
    deq = vals * scale[..., None]
    err = np.abs(deq - x.reshape(2, 64, 8, 32).astype(np.float64))
    # half an E4M3 ulp: 2^-4 relative for normals, 2^-10 * scale absolute for subnormals
    bound = np.maximum(np.abs(x.reshape(2, 64, 8, 32)) * 2.0 ** -4, 2.0 ** -10 * scale[..., None])
    assert np.all(err <= bound)


def test_mxfp8_exact_values_roundtrip():
    rng = np.random.default_rng(6)
    codes = rng.integers(0, 0x7E, (4, 32))
    e = rng.integers(-10, 10, (4, 1))
    vals = formats.decode_e4m3(codes) * np.exp2(e.astype(float))
    vals[:, 0] = 448.0 * np.exp2(e[:, 0].astype(float))  # the block max sits at the top code
    q, sf = quantize.quantize_logical(vals.astype(np.float32)[None], "mxfp8")
    assert np.array_equal(formats.decode_e4m3(q[0]) * formats.decode_e8m0(sf[0]), vals)


def test_nvfp4_quantiser_invariants():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((1, 32, 128)).astype(np.float32)
    codes, sf = quantize.quantize_logical(x, "nvfp4")
    s = formats.decode_ue4m3(sf)
    amax = np.abs(x.reshape(1, 32, 8, 16)).max(-1).astype(np.float64)
    # scale within half a UE4M3 ulp of amax/6 (relative 2^-4 in the normal range)
    assert np.all(np.abs(s - amax / 6) <= (amax / 6) * 2.0 ** -4 + 2.0 ** -10)
    vals = quantize.decode_codes(codes, "nvfp4").reshape(1, 32, 8, 16)
    q = x.reshape(1, 32, 8, 16) / s[..., None]
    grid = formats.E2M1_GRID
    # each code is a nearest grid point of x/s (clamped at 6)
    d_best = np.min(np.abs(np.minimum(np.abs(q), 6)[..., None] - grid), axis=-1)
    assert np.allclose(np.abs(np.abs(vals) - np.minimum(np.abs(q), 6)), d_best, atol=1e-12)


def test_dequantize_ragged_rows_and_batch():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((2, 130, 64)).astype(np.float32)
    for fmt in ("mxfp8", "nvfp4"):
        codes, sf = quantize.quantize(x, fmt)
        deq = quantize.dequantize(codes, sf, fmt, 130, 64, 2)
        codes_l, sf_l = quantize.quantize_logical(x, fmt)
        v = 32 if fmt == "mxfp8" else 16
        ref = quantize.decode_codes(codes_l, fmt) * np.repeat(quantize.decode_scales(sf_l, fmt), v, -1)
        assert np.array_equal(deq, ref)
        rows = np.array([0, 129, 130 + 7, 259])
        sub = quantize.dequantize_rows(codes.reshape(260, -1)[rows], sf, fmt, rows, 130, 64)
        assert np.array_equal(sub, deq.reshape(260, 64)[rows])

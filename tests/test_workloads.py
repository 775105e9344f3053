"""The seeded input generators: the properties the parity tests and the bench rely on.

The sampled full-size checks regenerate single rows of multi-gigabyte operands, so rows drawn
alone must equal the same rows of the whole tensor; expert row ranges must be the documented
256-padded cumulative ends; padding rows carry zeros; the RoPE tables follow their recipe.
"""
import numpy as np

import workloads as W


def test_rows_drawn_alone_equal_the_whole_tensor():
    rows, k = 37, 40000  # rows that straddle the 2^20-value chunks of the generator
    full = W.normal_f32(3, W.S_A, 0, rows * k).reshape(rows, k)
    pick = np.array([0, 5, 26, 36, 13])
    np.testing.assert_array_equal(W.normal_f32_rows(3, W.S_A, pick, k), full[pick])
    # different streams and seeds give different values
    assert not np.array_equal(W.normal_f32(3, W.S_B, 0, 1000), full.ravel()[:1000])
    assert not np.array_equal(W.normal_f32(4, W.S_A, 0, 1000), full.ravel()[:1000])


def test_workload_rows_match_their_full_operands():
    wl = W.Grouped("t", 3, 96, 64, 500, "fixed:200,0,300", "bf16", seed=2)
    a, b = wl.a_rows(), wl.b_rows()
    rows = np.array([0, 199, 200, 300, 767])
    np.testing.assert_array_equal(wl.a_rows(rows), a[rows])
    np.testing.assert_array_equal(wl.b_rows(np.array([0, 64, 191])), b.reshape(-1, 96)[[0, 64, 191]])
    d = W.Dense("t", 130, 70, 64, 2, "mxfp8", "f32", boost_every=7, seed=1)
    np.testing.assert_array_equal(d.a_rows(np.array([1, 131, 259])), d.a_rows().reshape(-1, 64)[[1, 131, 259]])


def test_expert_ranges_and_padding_rows():
    for wl in (W.GROUPED_SRELU_E32, W.GROUPED_FP8D_E128, W.GROUPED_FP8D_E32):
        counts = wl.counts()
        assert counts.sum() == wl.routed_rows and np.all(counts >= 0)
        ends = wl.padded_offsets().astype(np.int64)
        sizes = np.diff(np.concatenate([[0], ends]))
        assert np.all(ends % 256 == 0) and np.all(sizes >= counts) and np.all(sizes - counts < 256)
        assert wl.valid_m == ends[-1]
        mask = wl.routed_mask()
        assert mask.sum() == wl.routed_rows
    g = W.GroupedDswiglu("t", 3, 64, 32, 300, "fixed:10,0,290", "bf16", seed=1)
    mask = g.routed_mask()
    a, c = g.a_rows(), g.c_rows()
    assert np.all(a[~mask] == 0) and np.all(c[~mask] == 0) and np.any(c[mask] != 0)
    assert c.shape == (g.valid_m, 64)


def test_rope_tables():
    wl = W.RopeProj("t", 4100, 64, 1, 192, 64)
    cos, sin = wl.tables()
    assert cos.shape == sin.shape == (4100, 64)
    np.testing.assert_array_equal(cos[:, :32], cos[:, 32:])  # the same angle in both halves
    np.testing.assert_allclose(cos ** 2 + sin ** 2, 1.0, atol=1e-6)
    assert np.all(cos[0] == 1.0) and np.all(sin[0] == 0.0)
    np.testing.assert_array_equal(cos[W.SEQ_LEN_ROPE], cos[0])  # positions restart per sequence
    np.testing.assert_allclose(np.arctan2(sin[1, :32], cos[1, :32]), 10000.0 ** (-2.0 * np.arange(32) / 64),
                               rtol=1e-6)

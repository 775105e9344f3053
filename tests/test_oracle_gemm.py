"""Pins of the dense and grouped oracle against closed forms, brute force and invariants."""
import math

import numpy as np
import pytest

from oracle import formats, gemm, quantize, sf_layout


def _ones_operands(fmt, rows, k, batch, scale_code):
    v = 32 if fmt == "mxfp8" else 16
    if fmt == "mxfp8":
        codes = np.full((batch, rows, k), 0x38, np.uint8)       # E4M3 1.0
    else:
        codes = np.full((batch, rows, k // 2), 0x22, np.uint8)  # two E2M1 1.0 nibbles
    sf = sf_layout.pack(np.full((batch, rows, k // v), scale_code, np.uint8))
    return codes, sf


@pytest.mark.parametrize("fmt,sfa_code,sfb_code,sa,sb", [
    ("mxfp8", 127 + 3, 127 - 2, 2.0 ** 3, 2.0 ** -2),
    ("nvfp4", 0x40, 0x30, 2.0, 0.5),  # UE4M3 2.0 and 0.5
])
def test_dense_all_ones_closed_form(fmt, sfa_code, sfb_code, sa, sb):
    m, n, k, l = 130, 128, 256, 2
    a, sfa = _ones_operands(fmt, m, k, l, sfa_code)
    b, sfb = _ones_operands(fmt, n, k, l, sfb_code)
    c, amax = gemm.dense_gemm_amax(a, b, sfa, sfb, fmt, m, n, k, l)
    assert c.shape == (l, m, n)
    assert np.all(c == k * sa * sb) and amax == k * sa * sb


def test_dense_one_hot_rows_gather_b():
    m, n, k, l = 128, 128, 128, 1
    rng = np.random.default_rng(0)
    b, sfb = quantize.quantize(rng.standard_normal((l, n, k)).astype(np.float32), "mxfp8")
    a = np.zeros((l, m, k), np.uint8)
    picks = rng.integers(0, k, m)
    a[0, np.arange(m), picks] = 0x38                     # one 1.0 per row
    sfa = sf_layout.pack(np.full((l, m, k // 32), 127, np.uint8))
    c, _ = gemm.dense_gemm_amax(a, b, sfa, sfb, "mxfp8", m, n, k, l)
    bhat = quantize.dequantize(b, sfb, "mxfp8", n, k, l)
    assert np.array_equal(c[0], bhat[0][:, picks].T)


def _bruteforce_dense(a_codes, b_codes, sfa, sfb, fmt, m, n, k, l):
    """Scalar loops over the physical (L, MT, KT, 32, 4, 4) scale bytes (no offset formula)."""
    v = 32 if fmt == "mxfp8" else 16
    dec = formats.decode_e8m0 if fmt == "mxfp8" else formats.decode_ue4m3

    def scales(buf, rows):
        mt_n, kt_n = -(-rows // 128), -(-(k // v) // 4)
        phys = np.asarray(buf).reshape(l, mt_n, kt_n, 32, 4, 4)
        s = np.zeros((l, rows, k // v))
        for ll in range(l):
            for mt in range(mt_n):
                for kt in range(kt_n):
                    for i0 in range(32):
                        for i1 in range(4):
                            for k0 in range(4):
                                r, kb = mt * 128 + i1 * 32 + i0, kt * 4 + k0
                                if r < rows and kb < k // v:
                                    s[ll, r, kb] = dec(phys[ll, mt, kt, i0, i1, k0])
        return s

    def values(codes, rows):
        if fmt == "mxfp8":
            return formats.decode_e4m3(codes)
        out = np.zeros((l, rows, k))
        for j in range(k):
            byte = codes[..., j // 2]
            out[..., j] = formats.decode_e2m1((byte >> 4) if j % 2 else (byte & 0xF))
        return out

    sa, sb = scales(sfa, m), scales(sfb, n)
    av, bv = values(a_codes, m), values(b_codes, n)
    c = np.zeros((l, m, n))
    for ll in range(l):
        for i in range(m):
            for j in range(n):
                acc = 0.0
                for kk in range(k):
                    acc += av[ll, i, kk] * sa[ll, i, kk // v] * bv[ll, j, kk] * sb[ll, j, kk // v]
                c[ll, i, j] = acc
    return c


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_dense_bruteforce_tiny(fmt):
    m, n, k, l = 136, 5, 64, 2  # rows straddle two atoms; K = 2 (MXFP8) or 4 (NVFP4) blocks
    rng = np.random.default_rng(1)
    a, sfa = quantize.quantize(rng.standard_normal((l, m, k)).astype(np.float32) * 3, fmt)
    b, sfb = quantize.quantize(rng.standard_normal((l, n, k)).astype(np.float32), fmt)
    c, amax = gemm.dense_gemm_amax(a, b, sfa, sfb, fmt, m, n, k, l)
    ref = _bruteforce_dense(a, b, sfa, sfb, fmt, m, n, k, l)
    assert np.allclose(c, ref, rtol=0, atol=1e-12 * np.abs(ref).max())
    assert amax == np.max(np.abs(c))


def test_bruteforce_catches_transposed_scale_layout():
    """Planted mistake: swapping the i0/i1 roles of the atom changes the result."""
    m, n, k, l = 128, 4, 64, 1
    rng = np.random.default_rng(2)
    a, sfa = quantize.quantize(rng.standard_normal((l, m, k)).astype(np.float32) * np.exp2(rng.integers(-5, 5, (l, m, 1))), "mxfp8")
    b, sfb = quantize.quantize(rng.standard_normal((l, n, k)).astype(np.float32), "mxfp8")
    good = _bruteforce_dense(a, b, sfa, sfb, "mxfp8", m, n, k, l)
    bad_sfa = np.asarray(sfa).reshape(1, 1, 1, 32, 4, 4)[:, :, :, :, :, :].copy()
    bad_sfa = bad_sfa.reshape(1, 1, 1, 4, 32, 4).transpose(0, 1, 2, 4, 3, 5).copy().ravel()  # wrong row order
    c_bad, _ = gemm.dense_gemm_amax(a, b, bad_sfa, sfb, "mxfp8", m, n, k, l)
    assert not np.allclose(c_bad, good)


def _grouped_case(counts, k=64, n=64, fmt="mxfp8", seed=3):
    rng = np.random.default_rng(seed)
    pad = (np.asarray(counts) + 255) // 256 * 256
    offs = np.cumsum(pad).astype(np.int32)
    vm = int(offs[-1]) if len(offs) else 0
    x = rng.standard_normal((1, vm, k)).astype(np.float32)
    a, sfa = quantize.quantize(x, fmt)
    b, sfb = quantize.quantize(rng.standard_normal((len(counts), n, k)).astype(np.float32), fmt)
    alpha = rng.uniform(0.5, 2, len(counts)).astype(np.float32)
    prob = rng.uniform(0, 1, vm).astype(np.float32)
    return a, b, sfa, sfb, offs, alpha, prob, vm


def test_grouped_equals_per_expert_dense():
    counts = [0, 300, 0, 0, 1, 256, 0]  # empty experts first, in a run, and last
    k, n = 64, 64
    a, b, sfa, sfb, offs, alpha, prob, vm = _grouped_case(counts, k, n)
    c = gemm.grouped_gemm(a, b, sfa, sfb, "mxfp8", offs, alpha, k, n)
    ahat = quantize.dequantize(a, sfa, "mxfp8", vm, k, 1)[0]
    bhat = quantize.dequantize(b, sfb, "mxfp8", n, k, len(counts))
    begin = 0
    for g, end in enumerate(offs):
        rows = slice(begin, end)
        if end > begin:
            # an independent path: the dense oracle on this expert's rows with L = 1
            cg, _ = gemm.dense_gemm_amax(a[:, rows], b[g:g + 1], sf_layout.pack(
                sf_layout.unpack(sfa, vm, k // 32)[:, rows]), sf_layout.pack(
                sf_layout.unpack(sfb, n, k // 32, len(counts))[g:g + 1]), "mxfp8", end - begin, n, k, 1)
            assert np.allclose(c[rows], alpha[g] * cg[0], rtol=1e-14, atol=0)
            assert np.allclose(c[rows], alpha[g] * (ahat[rows] @ bhat[g].T), rtol=1e-14, atol=0)
        begin = end
    assert gemm.per_expert_amax(c, offs)[0] == 0 and gemm.per_expert_amax(c, offs)[-1] == 0


def test_expert_of_rows():
    offs = np.array([0, 256, 256, 768, 768], np.int32)
    g = gemm.expert_of_rows(offs, 768)
    assert np.all(g[:256] == 1) and np.all(g[256:] == 3)


def test_srelu_negative_c_gives_zero():
    counts = [256, 256]
    k, n = 64, 32
    rng = np.random.default_rng(4)
    x = rng.standard_normal((1, 512, k)).astype(np.float32)
    a, sfa = quantize.quantize(x, "mxfp8")
    # B rows equal to minus A rows: C[m, m'] = -<a_m, a_m'>, and C[m, m] < 0
    b_src = -x[0, :n][None].repeat(2, 0)
    b, sfb = quantize.quantize(b_src, "mxfp8")
    offs = np.array([256, 512], np.int32)
    out = gemm.grouped_srelu(a, b, sfa, sfb, "mxfp8", offs, np.ones(2, np.float32), np.ones(512, np.float32), k, n)
    diag = out["d"][np.arange(n), np.arange(n)]
    assert np.all(out["c"][np.arange(n), np.arange(n)] < 0) and np.all(diag == 0)
    assert np.all(out["d"][out["c"] <= 0] == 0)


def test_tanh_clamp_bounds_and_limits():
    c = np.linspace(-50, 5000, 20001).reshape(-1, 1) * np.ones((1, 3))
    prob = np.linspace(0, 1, c.shape[0])
    s = 32.0
    d = gemm.srelu(c, prob, s)
    assert np.all(d <= s * s * prob[:, None] * (1 + 1e-15))
    big = c[:, 0] > 40 * s
    assert np.allclose(d[big, 0], s * s * prob[big], rtol=1e-12)
    # s -> infinity reduces to the unclamped form
    small = gemm.srelu(c[:200], prob[:200], 1e12)
    assert np.allclose(small, gemm.srelu(c[:200], prob[:200]), rtol=1e-9)
    # unclamped is exactly prob * relu(c)^2
    assert np.array_equal(gemm.srelu(c, prob), prob[:, None] * np.maximum(c, 0) ** 2)


def test_fp8_d_requant_invariants():
    counts = [200, 0, 300]
    k, n = 64, 96
    a, b, sfa, sfb, offs, alpha, prob, vm = _grouped_case(counts, k, n, seed=9)
    for nc in (1.0, 0.75):
        out = gemm.grouped_srelu(a, b, sfa, sfb, "mxfp8", offs, alpha, prob, k, n, d_fp8=True, norm_const=nc)
        d = out["d"]
        for key, sfk, axis in (("d_row", "sfd_row_logical", 1), ("d_col", "sfd_col_logical", 0)):
            codes, sf = out[key], out[sfk]
            scale = formats.decode_e8m0(sf)
            vals = formats.decode_e4m3(codes)
            if axis == 1:
                deq = vals * np.repeat(scale, 32, axis=1) / nc
            else:
                deq = (vals.T * np.repeat(scale, 32, axis=1)).T / nc
            # dequantised D within half an E4M3 ulp of D (relative 2^-4, abs 2^-10*scale)
            sc = np.repeat(scale, 32, axis=1) if axis == 1 else np.repeat(scale, 32, axis=1).T
            assert np.all(np.abs(deq - d) <= np.maximum(np.abs(d) * 2.0 ** -4, 2.0 ** -10 * sc / nc) * (1 + 1e-12))
            blk = np.abs(vals if axis == 1 else vals.T).reshape(-1, 32).max(-1)
            nz = np.abs(d if axis == 1 else d.T).reshape(-1, 32).max(-1) > 0
            assert np.all((blk[nz] >= 224) & (blk[nz] <= 448))
        # physical buffers hold the logical scales
        assert np.array_equal(sf_layout.unpack(out["sfd_row"], vm, n // 32), out["sfd_row_logical"][None])
        assert np.array_equal(sf_layout.unpack(out["sfd_col"], n, vm // 32), out["sfd_col_logical"][None])


def test_workload_recipes():
    import workloads as W
    g = W.GROUPED_SRELU_E32
    offs = g.padded_offsets()
    assert offs.dtype == np.int32 and np.all(offs % 256 == 0) and np.all(np.diff(offs) >= 0)
    assert g.counts().sum() == 32768 and g.valid_m == offs[-1]
    z = W.GROUPED_FP8D_E128
    c = z.counts()
    assert c.sum() == 65536 and c[0] == c.max()
    d = W.DENSE_MXFP8_256
    a = d.a_rows()
    assert a.shape == (1, 256, 256) and a.dtype == np.float32
    assert np.array_equal(d.a_rows(np.array([5, 200])), a[0, [5, 200]])
    big = W.DENSE_MXFP8_8192
    rows = np.array([0, 8191, 3 * 8192 + 17])
    sub = big.a_rows(rows)
    assert sub.shape == (3, 8192)
    kb = np.arange(8192) // 32
    boosted = sub[:, kb % 7 == 6]
    plain = sub[:, kb % 7 != 6]
    assert np.abs(boosted).mean() > 30 * np.abs(plain).mean()
    assert math.isclose(float(np.std(plain)), 1.0, rel_tol=0.05)


def _bruteforce_abs_sum(a_codes, b_codes, sfa, sfb, fmt, m, n, k, l):
    """sum_k |a||sa| |b||sb| by scalar loops over the physical scale bytes (no offset formula, no matmul)."""
    v = 32 if fmt == "mxfp8" else 16
    dec = formats.decode_e8m0 if fmt == "mxfp8" else formats.decode_ue4m3

    def scale_of(buf, rows, ll, r, kb):
        kt_n = -(-(k // v) // 4)
        mt_n = -(-rows // 128)
        phys = np.asarray(buf).reshape(l, mt_n, kt_n, 32, 4, 4)
        return float(dec(phys[ll, r // 128, kb // 4, r % 32, (r % 128) // 32, kb % 4]))

    def value_of(codes, ll, r, kk):
        if fmt == "mxfp8":
            return float(formats.decode_e4m3(codes[ll, r, kk]))
        byte = int(codes[ll, r, kk // 2])
        return float(formats.decode_e2m1((byte >> 4) if kk % 2 else (byte & 0xF)))

    out = np.zeros((l, m, n))
    for ll in range(l):
        for i in range(m):
            for j in range(n):
                acc = 0.0
                for kk in range(k):
                    x = value_of(a_codes, ll, i, kk) * scale_of(sfa, m, ll, i, kk // v)
                    y = value_of(b_codes, ll, j, kk) * scale_of(sfb, n, ll, j, kk // v)
                    acc += abs(x) * abs(y)
                out[ll, i, j] = acc
    return out


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_dense_abs_sum_bruteforce_tiny(fmt):
    """dense_abs_sum (the scale of every C / D tolerance) against scalar loops on a ragged case
    with mixed signs and a 2^+-8 spread of block magnitudes."""
    m, n, k, l = 7, 5, 64, 2
    rng = np.random.default_rng(11)
    xa = rng.standard_normal((l, m, k)) * np.exp2(rng.integers(-8, 9, (l, m, 1)))
    xb = rng.standard_normal((l, n, k))
    a, sfa = quantize.quantize(xa.astype(np.float32), fmt)
    b, sfb = quantize.quantize(xb.astype(np.float32), fmt)
    s = gemm.dense_abs_sum(a, b, sfa, sfb, fmt, m, n, k, l)
    ref = _bruteforce_abs_sum(a, b, sfa, sfb, fmt, m, n, k, l)
    assert s.shape == (l, m, n)
    assert np.allclose(s, ref, rtol=1e-13, atol=0)
    c, _ = gemm.dense_gemm_amax(a, b, sfa, sfb, fmt, m, n, k, l)
    # the sum of magnitudes bounds |C| and, with mixed signs, is strictly larger somewhere
    assert np.all(np.abs(c) <= s * (1 + 1e-14)) and np.any(np.abs(c) < 0.9 * s)


@pytest.mark.parametrize("fmt,sfa_code,sfb_code,sa,sb", [
    ("mxfp8", 127 + 4, 127 - 3, 2.0 ** 4, 2.0 ** -3),
    ("nvfp4", 0x48, 0x28, 4.0, 0.25),  # UE4M3 4.0 and 0.25
])
def test_dense_abs_sum_signed_ones_closed_form(fmt, sfa_code, sfb_code, sa, sb):
    """Codes +-1 with random signs and scales 2^ea, 2^eb: sum_k |Ahat||Bhat| = K 2^(ea+eb) exactly,
    whatever the signs, while C (the signed sum) is smaller wherever signs disagree."""
    m, n, k, l = 130, 3, 256, 2
    rng = np.random.default_rng(12)
    a, sfa = _ones_operands(fmt, m, k, l, sfa_code)
    b, sfb = _ones_operands(fmt, n, k, l, sfb_code)
    if fmt == "mxfp8":
        a = a | (rng.integers(0, 2, a.shape) << 7).astype(np.uint8)   # sign bit of E4M3
        b = b | (rng.integers(0, 2, b.shape) << 7).astype(np.uint8)
    else:
        # sign bits of both E2M1 nibbles
        a = a | ((rng.integers(0, 2, a.shape) << 3) | (rng.integers(0, 2, a.shape) << 7)).astype(np.uint8)
        b = b | ((rng.integers(0, 2, b.shape) << 3) | (rng.integers(0, 2, b.shape) << 7)).astype(np.uint8)
    s = gemm.dense_abs_sum(a, b, sfa, sfb, fmt, m, n, k, l)
    assert np.all(s == k * sa * sb)
    c, _ = gemm.dense_gemm_amax(a, b, sfa, sfb, fmt, m, n, k, l)
    assert np.all(np.abs(c) < k * sa * sb)
    # planted mistake: the sum taken without the magnitudes is the signed C, which misses the closed form
    ahat = quantize.dequantize(a, sfa, fmt, m, k, l)
    bhat = quantize.dequantize(b, sfb, fmt, n, k, l)
    no_abs = np.matmul(ahat, np.swapaxes(bhat, -1, -2))
    assert not np.all(no_abs == k * sa * sb)


def _scalar_expert_max(d, padded_offsets):
    """Per-expert max |D| by a scan of every row (its expert found by a linear search of the ends)."""
    ends = [int(e) for e in padded_offsets]
    out = [0.0] * len(ends)
    for r in range(d.shape[0]):
        g = next(i for i, e in enumerate(ends) if r < e)
        for x in d[r]:
            out[g] = max(out[g], abs(float(x)))
    return np.array(out)


def _amax_case(seed=13):
    counts = [0, 300, 0, 0, 1, 256, 0]  # empty first, a run of empties, a 1-row expert, empty last
    pad = (np.asarray(counts) + 255) // 256 * 256
    offs = np.cumsum(pad).astype(np.int32)
    vm = int(offs[-1])
    rng = np.random.default_rng(seed)
    d = rng.standard_normal((vm, 24)) * np.exp2(rng.integers(-6, 7, (vm, 1)))
    # in every non-empty expert the largest magnitude is a negative entry
    begin = 0
    for end in offs:
        if end > begin:
            r = begin + (end - begin) // 3
            d[r, 5] = -2.0 * np.abs(d[begin:end]).max()
        begin = end
    return d, offs


def test_per_expert_amax_nonempty_experts():
    d, offs = _amax_case()
    got = gemm.per_expert_amax(d, offs)
    ref = _scalar_expert_max(d, offs)
    assert np.array_equal(got, ref)
    assert got[0] == 0 and got[2] == 0 and got[3] == 0 and got[-1] == 0 and np.all(got[[1, 4, 5]] > 0)
    # equal to the global max |D| over all rows, and to D's own maximum of the expert's rows
    assert got.max() == np.abs(d).max()


def test_per_expert_amax_catches_unadvanced_range():
    """Planted mistake: a scan whose range start is never advanced (every expert from row 0)
    disagrees with the scalar reference, so the pin above would catch it."""
    d, offs = _amax_case(seed=14)
    ref = _scalar_expert_max(d, offs)
    wrong = np.zeros(len(offs))
    for g, end in enumerate(offs):
        if end > 0:
            wrong[g] = np.abs(d[0:end]).max()
    assert not np.array_equal(wrong, ref)
    assert np.array_equal(gemm.per_expert_amax(d, offs), ref)

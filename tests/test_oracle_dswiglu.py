"""Pins of the dSwiGLU backward oracle ("Grouped GEMM + dSwiGLU (SM100)", Equations, Steps 1-3).

* the epilogue is the gradient of the forward SwiGLU: torch autograd (float64) through
  torch's own SiLU gives d/dx, d/dgate and d/dprob of sum(ref * prob * silu(gate) * x);
* closed forms at points where the sigmoid is known exactly (0, +-ln 3) and the limits
  of a saturated gate;
* the 32-column interleave against scalar loops and its round trip;
* the whole grouped path against per-element scalar evaluation on a tiny case, the
  identity prob * dprob = sum(ab * x), and (L, 2) amax with an empty expert.
"""
import math

import numpy as np
import pytest

from oracle import dswiglu, gemm, quantize


def test_epilogue_is_the_swiglu_gradient():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    rows, n = 7, 64
    ref = rng.standard_normal((rows, n)) * 3
    x = rng.standard_normal((rows, n)) * 2
    gate = rng.standard_normal((rows, n)) * 6
    gate[0, :8] = [-60.0, -30.0, -12.0, 0.0, 1e-9, 12.0, 30.0, 60.0]
    prob = rng.random(rows)
    ab, dsw, dprob = dswiglu.epilogue(ref, x, gate, prob)

    tx = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    tg = torch.tensor(gate, dtype=torch.float64, requires_grad=True)
    tp = torch.tensor(prob, dtype=torch.float64, requires_grad=True)
    tr = torch.tensor(ref, dtype=torch.float64)
    loss = (tr * tp[:, None] * torch.nn.functional.silu(tg) * tx).sum()
    loss.backward()
    np.testing.assert_allclose(ab, tx.grad.numpy(), rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(dsw, tg.grad.numpy(), rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(dprob, tp.grad.numpy(), rtol=1e-12, atol=0)


def test_epilogue_closed_forms():
    ln3 = math.log(3.0)
    ref, x, p = 2.0, -1.5, 0.25
    gate = np.array([[0.0, ln3, -ln3]])
    ab, dsw, dprob = dswiglu.epilogue(np.full((1, 3), ref), np.full((1, 3), x), gate, [p])
    sig = [0.5, 0.75, 0.25]
    for j in range(3):
        g, s = gate[0, j], sig[j]
        assert ab[0, j] == pytest.approx(ref * p * g * s, rel=1e-14, abs=1e-15)
        assert dsw[0, j] == pytest.approx(ref * p * x * s * (1 + g * (1 - s)), rel=1e-14)
    # gate 0: no swish, half the input gradient
    assert ab[0, 0] == 0.0 and dsw[0, 0] == pytest.approx(0.5 * ref * p * x, rel=1e-15)
    assert dprob[0] == pytest.approx(ref * x * (0.75 * ln3 - 0.25 * ln3), rel=1e-14)


def test_sigmoid_saturates_without_overflow():
    with np.errstate(over="raise", invalid="raise", divide="raise"):
        s = dswiglu.sigmoid(np.array([-1e4, -800.0, 0.0, 800.0, 1e4]))
    assert s[0] == 0.0 and s[-1] == 1.0 and s[2] == 0.5
    g = np.linspace(-40, 40, 161)
    np.testing.assert_allclose(dswiglu.sigmoid(-g), 1.0 - dswiglu.sigmoid(g), rtol=0, atol=4e-16)  # 1 - s rounds
    scipy_special = pytest.importorskip("scipy.special")
    np.testing.assert_allclose(dswiglu.sigmoid(g), scipy_special.expit(g), rtol=1e-15)
    # a saturated gate passes the gradient straight through (sig -> 1) or blocks it (sig -> 0)
    ab, dsw, _ = dswiglu.epilogue(np.ones((1, 2)), np.ones((1, 2)), np.array([[200.0, -200.0]]), [1.0])
    assert dsw[0, 0] == 1.0 and ab[0, 0] == 200.0
    assert abs(dsw[0, 1]) < 1e-80 and abs(ab[0, 1]) < 1e-80


def test_interleave_against_scalar_loops():
    rng = np.random.default_rng(2)
    rows, n = 3, 96
    c2 = rng.standard_normal((rows, 2 * n))
    x, gate = dswiglu.deinterleave(c2)
    for m in range(rows):
        for col in range(n):
            j, i = divmod(col, 32)
            assert x[m, col] == c2[m, 64 * j + i]
            assert gate[m, col] == c2[m, 64 * j + 32 + i]
    assert np.array_equal(dswiglu.interleave(x, gate), c2)
    d = dswiglu.interleave(np.zeros((rows, n)), np.ones((rows, n)))
    assert np.array_equal(d[0], np.tile(np.repeat([0.0, 1.0], 32), n // 32))


def test_grouped_path_scalar_and_invariants():
    rng = np.random.default_rng(3)
    k, n = 64, 64
    offs = np.array([256, 256, 512], dtype=np.int32)          # expert 1 is empty
    vm = 512
    a = (rng.standard_normal((1, vm, k)) / 8).astype(np.float32)
    b = (rng.standard_normal((3, n, k)) / 8).astype(np.float32)
    qa, sfa = quantize.quantize(a, "mxfp8")
    qb, sfb = quantize.quantize(b, "mxfp8")
    alpha = np.array([0.5, 3.0, 1.25])
    beta = np.array([2.0, 7.0, 0.75])
    prob = rng.random(vm)
    c_in = rng.standard_normal((vm, 2 * n)) * 3
    out = dswiglu.grouped_dswiglu(qa[0], qb, sfa, sfb, "mxfp8", offs, alpha, beta, prob, c_in, k, n)

    ahat = quantize.dequantize(qa, sfa, "mxfp8", vm, k, 1)[0]
    bhat = quantize.dequantize(qb, sfb, "mxfp8", n, k, 3)
    for m, col in [(0, 0), (17, 31), (255, 32), (256, 5), (300, 63), (511, 40)]:
        g = 0 if m < 256 else 2
        ref = alpha[g] * sum(float(ahat[m, kk]) * float(bhat[g, col, kk]) for kk in range(k))
        j, i = divmod(col, 32)
        xv = beta[g] * c_in[m, 64 * j + i]
        gv = beta[g] * c_in[m, 64 * j + 32 + i]
        sig = 1.0 / (1.0 + math.exp(-gv))
        ab = ref * prob[m] * gv * sig
        dsw = ref * prob[m] * xv * sig * (1.0 + gv * (1.0 - sig))
        assert out["ref"][m, col] == pytest.approx(ref, rel=1e-12, abs=1e-14)
        assert out["d"][m, 64 * j + i] == pytest.approx(ab, rel=1e-10, abs=1e-14)
        assert out["d"][m, 64 * j + 32 + i] == pytest.approx(dsw, rel=1e-10, abs=1e-14)
    # prob * dprob = sum_n ab * x
    np.testing.assert_allclose(prob * out["dprob"], np.sum(out["ab"] * out["x"], axis=1), rtol=1e-12, atol=1e-14)
    # ref is the grouped GEMM of the sReLU path
    np.testing.assert_array_equal(out["ref"], gemm.grouped_gemm(qa[0], qb, sfa, sfb, "mxfp8", offs, alpha, k, n))
    amax = out["amax"]
    assert amax.shape == (3, 2) and np.all(amax[1] == 0)
    assert amax[0, 0] == np.abs(out["d"][:256].reshape(256, -1, 2, 32)[:, :, 0]).max()
    assert amax[2, 1] == np.abs(out["d"][256:].reshape(256, -1, 2, 32)[:, :, 1]).max()


def test_grouped_fp8_outputs_cover_2n_columns():
    rng = np.random.default_rng(4)
    k, n, vm = 64, 32, 256
    qa, sfa = quantize.quantize((rng.standard_normal((1, vm, k)) / 8).astype(np.float32), "mxfp8")
    qb, sfb = quantize.quantize((rng.standard_normal((1, n, k)) / 8).astype(np.float32), "mxfp8")
    out = dswiglu.grouped_dswiglu(qa[0], qb, sfa, sfb, "mxfp8", np.array([vm], np.int32), [1.0], [1.0],
                                  rng.random(vm), rng.standard_normal((vm, 2 * n)), k, n, d_fp8=True,
                                  norm_const=0.5)
    assert out["d_row"].shape == (vm, 2 * n) and out["d_col"].shape == (vm, 2 * n)
    assert out["sfd_row_logical"].shape == (vm, 2) and out["sfd_col_logical"].shape == (2 * n, vm // 32)
    # the row scales of the ab and dswiglu blocks are those of each block on its own
    row_codes, row_sf = gemm.mxfp8_quantize_blocks(out["ab"], 0.5, axis=1)
    assert np.array_equal(row_sf[:, 0], out["sfd_row_logical"][:, 0])
    assert np.array_equal(row_codes, out["d_row"][:, :32])

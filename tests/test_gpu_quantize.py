"""GPU parity of bsg_quantize_mx (fp32 input) and bsg_quantize_mx_bf16 (bf16 input) against the oracle
quantiser: codes and scale bytes bit-exact."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats, quantize as oq

pytestmark = pytest.mark.gpu


def _wide_range(seed, batch, rows, k, v):
    """N(0,1) values with a per-block power-of-two spread of 2^-40 .. 2^40 and some zero blocks."""
    x = W.normal_f32(seed, 11, 0, batch * rows * k).reshape(batch, rows, k)
    e = W.normal_f32(seed, 12, 0, batch * rows * (k // v)).reshape(batch, rows, k // v)
    e = np.clip(np.round(e * 12), -40, 40).astype(np.float32)
    x = x * np.repeat(np.exp2(e), v, axis=-1).astype(np.float32)
    x[..., :v][np.abs(e[..., 0]) > 25] = 0.0  # a few all-zero blocks
    return x.astype(np.float32)


def _ties(fmt, batch, rows, k):
    """Values sitting exactly on rounding midpoints of the code grid (after the block scale)."""
    rng_vals = W.normal_f32(5, 13, 0, batch * rows * k).reshape(batch, rows, k)
    if fmt == "mxfp8":
        grid = formats.decode_e4m3(np.arange(0, 0x7F))
        mids = (grid[:-1] + grid[1:]) / 2
        idx = (np.abs(rng_vals) * 1000).astype(np.int64) % len(mids)
        x = np.where(rng_vals < 0, -mids[idx], mids[idx])
        x[..., ::32] = 448.0  # pins every block's scale to 2^0
    else:
        mids = formats.E2M1_MIDS
        idx = (np.abs(rng_vals) * 1000).astype(np.int64) % len(mids)
        x = np.where(rng_vals < 0, -mids[idx], mids[idx])
        x[..., ::16] = 6.0  # block scale 1.0
    return x.astype(np.float32)


def _run(lib, x, fmt):
    from nvfp4_gemm_moe_gb300 import torch_ops
    xg = torch.from_numpy(x).cuda()
    q, sf = torch_ops.quantize(xg, fmt)
    torch.cuda.synchronize()
    return q.cpu().numpy(), sf.cpu().numpy()


@pytest.mark.parametrize("fmt,batch,rows,k", [
    ("mxfp8", 1, 256, 256), ("mxfp8", 2, 130, 160), ("mxfp8", 1, 1, 32), ("mxfp8", 3, 129, 4096),
    ("nvfp4", 1, 256, 512), ("nvfp4", 2, 130, 96), ("nvfp4", 1, 3, 32), ("nvfp4", 2, 200, 2080),
])
def test_quantize_bit_exact_wide_range(lib, fmt, batch, rows, k):
    v = 32 if fmt == "mxfp8" else 16
    x = _wide_range(batch * 1000 + rows + k, batch, rows, k, v)
    q, sf = _run(lib, x, fmt)
    q_ref, sf_ref = oq.quantize(x, fmt)
    assert np.array_equal(sf, sf_ref), f"{(sf != sf_ref).sum()} scale bytes differ"
    assert np.array_equal(q.reshape(q_ref.shape), q_ref), f"{(q.reshape(q_ref.shape) != q_ref).sum()} code bytes differ"


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_quantize_bit_exact_ties(lib, fmt):
    x = _ties(fmt, 2, 128, 256)
    q, sf = _run(lib, x, fmt)
    q_ref, sf_ref = oq.quantize(x, fmt)
    assert np.array_equal(sf, sf_ref)
    assert np.array_equal(q.reshape(q_ref.shape), q_ref)


def test_quantize_nvfp4_scale_ties_and_saturation(lib):
    """Block maxima at 6 * (E4M3 midpoints) test the exact scale rounding; huge maxima saturate."""
    grid = formats.decode_e4m3(np.arange(0, 0x7F))
    mids = (grid[:-1] + grid[1:]) / 2
    amax = np.concatenate([6 * mids, [3000.0, 1e6, 6 * 2.0 ** -11, 6 * 2.0 ** -10]]).astype(np.float32)
    amax = amax[np.abs(amax.astype(np.float64) - np.concatenate([6 * mids, [3000.0, 1e6, 6 * 2.0 ** -11,
                                                                           6 * 2.0 ** -10]])) == 0]
    rows = len(amax)
    x = np.zeros((1, rows, 32), np.float32)
    x[0, :, 0] = amax
    x[0, :, 1] = -amax * np.float32(0.3)
    x[0, :, 16] = amax * np.float32(0.5)
    q, sf = _run(lib, x, "nvfp4")
    q_ref, sf_ref = oq.quantize(x, "nvfp4")
    assert np.array_equal(sf, sf_ref)
    assert np.array_equal(q.reshape(q_ref.shape), q_ref)


def test_quantize_workload_rows_bit_exact(lib):
    """The recipe of the large batched dense workload (with its 2^6-boosted K blocks), on a row slice."""
    wl = W.DENSE_MXFP8_8192
    rows = np.arange(0, 256)
    x = wl.a_rows(rows)[None]
    q, sf = _run(lib, x, "mxfp8")
    q_ref, sf_ref = oq.quantize(x, "mxfp8")
    assert np.array_equal(sf, sf_ref) and np.array_equal(q.reshape(q_ref.shape), q_ref)


def test_quantize_nvfp4_near_midpoints(lib):
    """Values 1 to 80 ulps on either side of every E2M1 midpoint, under many block scales: the
    hardware-conversion fast path and its exact fallback must both agree with the oracle."""
    rng = np.random.default_rng(17)
    rows, k = 256, 512
    mids = np.asarray(formats.E2M1_MIDS, dtype=np.float32)
    n = rows * k
    m = mids[rng.integers(0, len(mids), n)]
    # even rows stay 40+ ulps of x (20+ of x / s) away, so their units take the fast path; odd
    # rows come within 1 ulp
    lo = np.where((np.arange(n) // k) % 2 == 0, 40, 1)
    ulps = (rng.integers(lo, 81) * rng.choice([-1, 1], n)).astype(np.int32)
    scale_codes = rng.integers(0x10, 0x70, rows * k // 16)  # UE4M3 scales 2^-5 .. 2^6 with mantissas
    s = np.repeat(formats.decode_ue4m3(scale_codes), 16).astype(np.float32)
    base = (m * s).astype(np.float32)  # exact: 3 + 4 significant bits
    x = (base.view(np.int32) + ulps).view(np.float32)
    x = np.where(rng.random(n) < 0.5, -x, x).astype(np.float32)
    # each block's amax (40 ulps above 6 s, so off the E2M1 grid) pins its scale to s
    pin = ((6.0 * s[::16]).astype(np.float32).view(np.int32) + 40).view(np.float32)
    x[::16] = np.copysign(pin, x[::16])
    x = x.reshape(1, rows, k)
    q, sf = _run(lib, x, "nvfp4")
    q_ref, sf_ref = oq.quantize(x, "nvfp4")
    assert np.array_equal(sf, sf_ref)
    assert np.array_equal(q.reshape(q_ref.shape), q_ref), f"{(q.reshape(q_ref.shape) != q_ref).sum()} code bytes differ"


@pytest.mark.parametrize("fmt,batch,rows,k", [
    ("mxfp8", 1, 256, 256), ("mxfp8", 2, 130, 160), ("mxfp8", 1, 1, 32), ("mxfp8", 3, 129, 4096),
    ("nvfp4", 1, 256, 512), ("nvfp4", 2, 130, 96), ("nvfp4", 1, 3, 32), ("nvfp4", 2, 200, 2080),
])
def test_quantize_bf16_input_bit_exact(lib, fmt, batch, rows, k):
    """bf16 input: the codes and scales the oracle gives for the (exactly widened) bf16 values,
    and the same bytes as the fp32 kernel on those values."""
    from nvfp4_gemm_moe_gb300 import torch_ops
    v = 32 if fmt == "mxfp8" else 16
    xb = torch.from_numpy(_wide_range(batch * 1000 + rows + k + 7, batch, rows, k, v)).to(torch.bfloat16)
    q, sf = torch_ops.quantize(xb.cuda(), fmt)
    q32, sf32 = torch_ops.quantize(xb.float().cuda(), fmt)
    torch.cuda.synchronize()
    q, sf = q.cpu().numpy(), sf.cpu().numpy()
    q_ref, sf_ref = oq.quantize(xb.float().numpy(), fmt)
    assert np.array_equal(sf, sf_ref), f"{(sf != sf_ref).sum()} scale bytes differ"
    assert np.array_equal(q.reshape(q_ref.shape), q_ref), f"{(q.reshape(q_ref.shape) != q_ref).sum()} code bytes differ"
    assert np.array_equal(q, q32.cpu().numpy()) and np.array_equal(sf, sf32.cpu().numpy())


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_quantize_bf16_input_ties(lib, fmt):
    """Values on rounding midpoints (all representable in bf16: at most five significant bits)."""
    from nvfp4_gemm_moe_gb300 import torch_ops
    x = _ties(fmt, 2, 130, 256)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(xb.float().numpy(), x)
    q, sf = torch_ops.quantize(xb.cuda(), fmt)
    torch.cuda.synchronize()
    q_ref, sf_ref = oq.quantize(x, fmt)
    assert np.array_equal(sf.cpu().numpy(), sf_ref)
    assert np.array_equal(q.cpu().numpy().reshape(q_ref.shape), q_ref)


def test_quantize_rejects_other_input_types(lib):
    from nvfp4_gemm_moe_gb300 import torch_ops
    with pytest.raises(TypeError):
        torch_ops.quantize(torch.zeros((1, 128, 64), dtype=torch.float16, device="cuda"), "mxfp8")


def test_quantize_bf16_nvfp4_exact_ties_under_uneven_scales(lib):
    """NVFP4 from bf16: values exactly on an E2M1 midpoint or code times a block scale that is not
    a power of two (so x * (1/s) is inexact and lands beside the tie), and their bf16 neighbours
    one unit away, which must round by value."""
    from nvfp4_gemm_moe_gb300 import torch_ops
    rng = np.random.default_rng(21)
    scales = np.array([1.125, 1.375, 1.75, 0.625, 2.5, 0.3125, 13.0, 0.0390625])  # UE4M3 values
    grid = np.array([0.5, 1.0, 1.5, 2.0, 3.0, 4.0])
    pts = np.concatenate([np.asarray(formats.E2M1_MIDS, dtype=np.float64), grid])
    rows, k = 256, 512
    nblk = k // 16
    s_blk = rng.choice(scales, (rows, nblk))
    x = rng.choice(pts, (rows, nblk, 16)) * s_blk[..., None]
    x[..., 0] = 6.0 * s_blk  # the block amax fixes the scale: RNE_UE4M3(amax / 6) = s
    x *= rng.choice([-1.0, 1.0], x.shape)
    xb = torch.from_numpy(x.reshape(rows, k).astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(xb.double().numpy(), x.reshape(rows, k))  # all exactly representable
    # a quarter of the non-amax values moved one bf16 unit up or down (no longer ties)
    bits = xb.view(torch.int16).numpy().copy().reshape(rows, nblk, 16)
    move = rng.random((rows, nblk, 16)) < 0.25
    move[..., 0] = False
    bits = np.where(move, bits + rng.choice(np.array([-1, 1], dtype=np.int16), bits.shape), bits).astype(np.int16)
    xb = torch.from_numpy(bits.reshape(rows, k)).view(torch.bfloat16)
    q, sf = torch_ops.quantize(xb.cuda(), "nvfp4")
    torch.cuda.synchronize()
    q_ref, sf_ref = oq.quantize(xb.float().numpy()[None], "nvfp4")
    assert np.array_equal(sf.cpu().numpy(), sf_ref)
    qg = q.cpu().numpy().reshape(q_ref.shape)
    assert np.array_equal(qg, q_ref), f"{(qg != q_ref).sum()} code bytes differ"

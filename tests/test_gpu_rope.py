"""GPU parity of bsg_gemm_rope_mxfp8 and bsg_gemm_rope_bf16 (projection GEMM + per-head RoPE + dual
MXFP8) against the oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats, quantize as oq, rope as orope
from guards import Outputs
from parity import TOL_C, check_e4m3_blocks

pytestmark = pytest.mark.gpu


def _tolerance(raw, s_abs, cos, sin, head_dim, qk_rope):
    """Bound on |Y_gpu - Y| per element (tokens, H, D) from the un-rotated projection ``raw`` and
    s_abs = sum_k |xhat||what|: the accumulation bound 2^-20 s_abs plus fp32 rounding on the
    no-position features; on the rotary ones that bound carried through the rotation (linear
    in a and b) plus the rounding of a product and a fused multiply-add."""
    p, half = head_dim - qk_rope, qk_rope // 2
    t = TOL_C * s_abs + 2.0 ** -22 * np.abs(raw)
    a, b = raw[..., p::2], raw[..., p + 1::2]
    ta, tb = TOL_C * s_abs[..., p::2], TOL_C * s_abs[..., p + 1::2]
    c1, c2 = np.abs(cos[:, None, :half]), np.abs(cos[:, None, half:])
    s1, s2 = np.abs(sin[:, None, :half]), np.abs(sin[:, None, half:])
    t[..., p:p + half] = c1 * ta + s1 * tb + 2.0 ** -22 * (np.abs(a) * c1 + np.abs(b) * s1)
    t[..., p + half:] = c2 * tb + s2 * ta + 2.0 ** -22 * (np.abs(b) * c2 + np.abs(a) * s2)
    return t


def run_rope(tokens, q_lora, heads, layout="atoms", seed=7, cta_pair=0, tile_n=0):
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg
    wl = W.RopeProj("t", tokens, q_lora, heads, 192, 64, seed=seed)
    x, w = wl.x_rows(), wl.w_rows()
    cos32, sin32 = wl.tables()
    cos = torch.from_numpy(cos32).to(torch.bfloat16)
    sin = torch.from_numpy(sin32).to(torch.bfloat16)
    qx, sx = torch_ops.quantize(torch.from_numpy(x).cuda(), "mxfp8")
    qw, sw = torch_ops.quantize(torch.from_numpy(w).cuda(), "mxfp8")
    xc, xs = oq.quantize_logical(x[None], "mxfp8")
    wc, wsc = oq.quantize_logical(w[None], "mxfp8")
    assert np.array_equal(qx[0].cpu().numpy(), xc[0]) and np.array_equal(qw[0].cpu().numpy(), wc[0])
    if layout == "plain":
        sx_in = torch.from_numpy(np.ascontiguousarray(xs[0])).cuda()
        sw_in = torch.from_numpy(np.ascontiguousarray(wsc[0])).cuda()
    else:
        sx_in, sw_in = sx, sw
    ws = torch.zeros(bsg.bsg_rope_workspace_size(tokens, heads, 192, q_lora), dtype=torch.uint8, device="cuda")
    g = Outputs()
    outputs = {"out_fp8_row": g.codes("row", (tokens, heads, 192)),
               "out_scales_row": g.scales("scales_row", (tokens, heads, 6)),
               "out_fp8_col": g.codes("col", (tokens, heads, 192)),
               "out_scales_col": g.scales("scales_col", (tokens // 32, heads, 192))}
    out = torch_ops.gemm_rope_mxfp8(qx[0], sx_in, qw[0], sw_in, cos.cuda(), sin.cuda(), heads, scale_layout=layout,
                                    workspace=ws, cta_pair=cta_pair, tile_n=tile_n, outputs=outputs)
    torch.cuda.synchronize()
    g.check()
    assert bsg.bsg_read_device_error(ws) == 0

    cos64, sin64 = cos.double().numpy(), sin.double().numpy()
    ref = orope.project(xc[0], xs[0], wc[0], wsc[0], cos64, sin64, heads, 192, 64)
    xh, wh = orope.dequantize_plain(xc[0], xs[0]), orope.dequantize_plain(wc[0], wsc[0])
    s_abs = (np.abs(xh) @ np.abs(wh).T).reshape(tokens, heads, 192)
    tol = _tolerance((xh @ wh.T).reshape(tokens, heads, 192), s_abs, cos64, sin64, 192, 64)
    n = heads * 192
    y = ref["y"].reshape(tokens, n)
    t = tol.reshape(tokens, n)
    check_e4m3_blocks(out["out_fp8_row"].cpu().numpy().reshape(tokens, n),
                      out["out_scales_row"].cpu().numpy().reshape(tokens, n // 32), y, t, 1.0, axis=1, what="row")
    check_e4m3_blocks(out["out_fp8_col"].cpu().numpy().reshape(tokens, n),
                      out["out_scales_col"].cpu().numpy().reshape(tokens // 32, n).T, y, t, 1.0, axis=0, what="col")
    return out, ref


@pytest.mark.parametrize("tokens,q_lora,heads,layout", [
    (128, 256, 1, "atoms"),
    (256, 512, 3, "atoms"),
    (384, 96, 5, "plain"),     # K below one 128-wide stage
    (512, 1536, 2, "plain"),
])
def test_gemm_rope(lib, tokens, q_lora, heads, layout):
    run_rope(tokens, q_lora, heads, layout)


@pytest.mark.parametrize("tokens,q_lora,heads,layout,cta_pair,tile_n", [
    (256, 256, 4, "atoms", 2, 0),     # CTA pairs on 256 x 256 tiles spanning heads
    (512, 160, 8, "plain", 2, 0),
    (256, 512, 4, "atoms", 1, 0),     # the same shape on one-CTA 128 x 192 tiles
    (256, 512, 4, "atoms", 2, 192),   # CTA pairs on 256 x 192 tiles, one head per CTA (automatic)
    (384, 256, 2, "atoms", 0, 0),     # automatic with tokens % 256 != 0: one-CTA tiles
    (512, 160, 3, "plain", 2, 192),   # N = 576: not a multiple of 256, fine for 192-wide pairs
    (768, 96, 5, "atoms", 2, 192),    # K below one stage
])
def test_gemm_rope_tile_shapes(lib, tokens, q_lora, heads, layout, cta_pair, tile_n):
    run_rope(tokens, q_lora, heads, layout, cta_pair=cta_pair, tile_n=tile_n)


def test_gemm_rope_identity_tables(lib):
    """cos = 1, sin = 0: the rotary features are the de-interleaved projection."""
    from nvfp4_gemm_moe_gb300 import torch_ops
    wl = W.RopeProj("t", 128, 128, 2, 192, 64, seed=3)
    qx, sx = torch_ops.quantize(torch.from_numpy(wl.x_rows()).cuda(), "mxfp8")
    qw, sw = torch_ops.quantize(torch.from_numpy(wl.w_rows()).cuda(), "mxfp8")
    ones = torch.ones((128, 64), dtype=torch.bfloat16, device="cuda")
    zeros = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    out = torch_ops.gemm_rope_mxfp8(qx[0], sx, qw[0], sw, ones, zeros, 2)
    # the same projection with the pair order undone on the host: rotary block codes are a
    # permutation of the un-rotated ones when the block scale is unchanged
    out0 = torch_ops.gemm_rope_mxfp8(qx[0], sx, qw[0], sw, ones, zeros, 2)
    torch.cuda.synchronize()
    assert torch.equal(out["out_fp8_row"], out0["out_fp8_row"])  # deterministic
    xc, xs = oq.quantize_logical(wl.x_rows()[None], "mxfp8")
    wc, wsc = oq.quantize_logical(wl.w_rows()[None], "mxfp8")
    ref = orope.project(xc[0], xs[0], wc[0], wsc[0], np.ones((128, 64)), np.zeros((128, 64)), 2, 192, 64)
    y = ref["y"]
    raw = (orope.dequantize_plain(xc[0], xs[0]) @ orope.dequantize_plain(wc[0], wsc[0]).T).reshape(128, 2, 192)
    np.testing.assert_array_equal(y[..., 128:160], raw[..., 128::2])
    np.testing.assert_array_equal(y[..., 160:], raw[..., 129::2])


def test_gemm_rope_validation(lib):
    """Invalid arguments are rejected on the host before anything is enqueued (real buffers, so
    a call that got through could not touch memory it does not own)."""
    import ctypes
    import nvfp4_gemm_moe_gb300 as bsg
    dev = "cuda"
    tokens, q_lora, heads = 256, 256, 2
    n = heads * 192
    x = torch.zeros((tokens, q_lora), dtype=torch.uint8, device=dev)
    w = torch.zeros((n, q_lora), dtype=torch.uint8, device=dev)
    sx = torch.zeros(bsg.bsg_sf_bytes(1, tokens, q_lora, 32), dtype=torch.uint8, device=dev)
    sw = torch.zeros(bsg.bsg_sf_bytes(1, n, q_lora, 32), dtype=torch.uint8, device=dev)
    tab = torch.zeros((tokens, 64), dtype=torch.bfloat16, device=dev)
    o_row = torch.zeros((tokens, heads, 192), dtype=torch.uint8, device=dev)
    s_row = torch.zeros((tokens, heads, 6), dtype=torch.uint8, device=dev)
    o_col = torch.zeros((tokens, heads, 192), dtype=torch.uint8, device=dev)
    s_col = torch.zeros((tokens // 32, heads, 192), dtype=torch.uint8, device=dev)
    ws = torch.zeros(bsg.bsg_workspace_size(), dtype=torch.uint8, device=dev)

    def call(cta_pair=0, **kw):
        a = dict(tokens=tokens, q_lora=q_lora, heads=heads, hd=192, rope=64, layout=0, wsb=ws.numel())
        a.update(kw)
        o = bsg._opts(cta_pair=cta_pair)
        return bsg.raw_status("bsg_gemm_rope_mxfp8", x.data_ptr(), sx.data_ptr(), w.data_ptr(), sw.data_ptr(),
                              a["layout"], tab.data_ptr(), tab.data_ptr(), a["tokens"], a["q_lora"], a["heads"],
                              a["hd"], a["rope"], o_row.data_ptr(), s_row.data_ptr(), o_col.data_ptr(),
                              s_col.data_ptr(), ctypes.byref(o), ws.data_ptr(), a["wsb"], None)
    assert call(tokens=100) == 1 and call(q_lora=48) == 1 and call(layout=2) == 1
    assert call(hd=128) == 2 and call(rope=32) == 2
    assert call(layout=1) == 8  # the plain layout needs room for the repacked scales
    assert call(cta_pair=2, tokens=128) == 1  # CTA pairs need tokens % 256 == 0 and heads * 192 % 256 == 0
    torch.cuda.synchronize()


def run_rope_bf16(tokens, q_lora, heads, seed=11, cta_pair=0):
    """The BF16-input path: the generator's fp32 values rounded to bf16 are the operands; the
    oracle takes those exact values."""
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg
    wl = W.RopeProj("t", tokens, q_lora, heads, 192, 64, seed=seed)
    x = torch.from_numpy(wl.x_rows()).to(torch.bfloat16)
    w = torch.from_numpy(wl.w_rows()).to(torch.bfloat16)
    cos32, sin32 = wl.tables()
    cos = torch.from_numpy(cos32).to(torch.bfloat16)
    sin = torch.from_numpy(sin32).to(torch.bfloat16)
    ws = torch.zeros(bsg.bsg_workspace_size(), dtype=torch.uint8, device="cuda")
    g = Outputs()
    outputs = {"out_fp8_row": g.codes("row", (tokens, heads, 192)),
               "out_scales_row": g.scales("scales_row", (tokens, heads, 6)),
               "out_fp8_col": g.codes("col", (tokens, heads, 192)),
               "out_scales_col": g.scales("scales_col", (tokens // 32, heads, 192))}
    out = torch_ops.gemm_rope_bf16(x.cuda(), w.cuda(), cos.cuda(), sin.cuda(), heads, workspace=ws, outputs=outputs,
                                   cta_pair=cta_pair)
    torch.cuda.synchronize()
    g.check()
    assert bsg.bsg_read_device_error(ws) == 0

    xh, wh = x.double().numpy(), w.double().numpy()
    cos64, sin64 = cos.double().numpy(), sin.double().numpy()
    ref = orope.project_bf16(xh, wh, cos64, sin64, heads, 192, 64)
    # bf16 x bf16 products are exact in fp32, as E4M3 ones are: the same accumulation bound
    s_abs = (np.abs(xh) @ np.abs(wh).T).reshape(tokens, heads, 192)
    tol = _tolerance((xh @ wh.T).reshape(tokens, heads, 192), s_abs, cos64, sin64, 192, 64)
    n = heads * 192
    y = ref["y"].reshape(tokens, n)
    t = tol.reshape(tokens, n)
    check_e4m3_blocks(out["out_fp8_row"].cpu().numpy().reshape(tokens, n),
                      out["out_scales_row"].cpu().numpy().reshape(tokens, n // 32), y, t, 1.0, axis=1, what="row")
    check_e4m3_blocks(out["out_fp8_col"].cpu().numpy().reshape(tokens, n),
                      out["out_scales_col"].cpu().numpy().reshape(tokens // 32, n).T, y, t, 1.0, axis=0, what="col")
    return out, ref


@pytest.mark.parametrize("tokens,q_lora,heads", [
    (128, 512, 1),
    (256, 1536, 3),    # the DeepSeek-V3 query down-projection rank
    (384, 72, 2),      # K tail of 8 values: one MMA with its upper half zero-filled
    (256, 232, 4),     # a partial last stage of three MMAs
    (512, 64, 8),      # a single 64-value K stage
])
def test_gemm_rope_bf16(lib, tokens, q_lora, heads):
    run_rope_bf16(tokens, q_lora, heads)


@pytest.mark.parametrize("tokens,q_lora,heads,cta_pair", [
    (256, 1536, 3, 2),   # CTA pairs on 256 x 192 tiles
    (512, 72, 2, 2),     # K tail of 8 values
    (256, 232, 5, 2),    # partial last stage
    (768, 64, 1, 2),     # one head, three pair tiles
    (256, 512, 2, 1),    # one-CTA tiles requested explicitly
])
def test_gemm_rope_bf16_tile_shapes(lib, tokens, q_lora, heads, cta_pair):
    run_rope_bf16(tokens, q_lora, heads, cta_pair=cta_pair)


def test_gemm_rope_bf16_matches_the_mxfp8_path_on_shared_values(lib):
    """Operands whose MXFP8 encoding is exact: the bf16 and MXFP8 kernels see the same values and
    must give identical codes and scales (both accumulate exact products in fp32, in the same
    K order up to the MMA grouping, so allow the boundary rule of the E4M3 check)."""
    from nvfp4_gemm_moe_gb300 import torch_ops
    tokens, q_lora, heads = 256, 256, 2
    rng = np.random.default_rng(5)
    grid = formats.decode_e4m3(np.arange(0, 0x7F, dtype=np.uint8))
    grid = grid[(grid >= 0.125) & (grid <= 8)]
    x = (rng.choice(grid, (tokens, q_lora)) * rng.choice([-1, 1], (tokens, q_lora))).astype(np.float32)
    w = (rng.choice(grid, (heads * 192, q_lora)) * rng.choice([-1, 1], (heads * 192, q_lora)) / 16).astype(np.float32)
    x[:, ::32] = 8.0
    w[:, ::32] = 0.5
    wl = W.RopeProj("t", tokens, q_lora, heads, 192, 64, seed=1)
    cos32, sin32 = wl.tables()
    cos = torch.from_numpy(cos32).to(torch.bfloat16).cuda()
    sin = torch.from_numpy(sin32).to(torch.bfloat16).cuda()
    qx, sx = torch_ops.quantize(torch.from_numpy(x).cuda(), "mxfp8")
    qw, sw = torch_ops.quantize(torch.from_numpy(w).cuda(), "mxfp8")
    a = torch_ops.gemm_rope_mxfp8(qx[0], sx, qw[0], sw, cos, sin, heads)
    b = torch_ops.gemm_rope_bf16(torch.from_numpy(x).to(torch.bfloat16).cuda(),
                                 torch.from_numpy(w).to(torch.bfloat16).cuda(), cos, sin, heads)
    torch.cuda.synchronize()
    ref = orope.project_bf16(x.astype(np.float64), w.astype(np.float64), cos.double().cpu().numpy(),
                             sin.double().cpu().numpy(), heads, 192, 64)
    s_abs = (np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64)).T).reshape(tokens, heads, 192)
    raw = (x.astype(np.float64) @ w.astype(np.float64).T).reshape(tokens, heads, 192)
    tol = _tolerance(raw, s_abs, cos.double().cpu().numpy(), sin.double().cpu().numpy(), 192, 64)
    n = heads * 192
    for out in (a, b):
        check_e4m3_blocks(out["out_fp8_row"].cpu().numpy().reshape(tokens, n),
                          out["out_scales_row"].cpu().numpy().reshape(tokens, n // 32), ref["y"].reshape(tokens, n),
                          tol.reshape(tokens, n), 1.0, axis=1, what="row")
    # the scales agree except where a block amax sits on a power-of-two boundary
    same = (a["out_scales_row"] == b["out_scales_row"]).float().mean().item()
    assert same > 0.99


def test_gemm_rope_bf16_validation(lib):
    """Invalid arguments are rejected before anything is enqueued (real buffers)."""
    import ctypes
    import nvfp4_gemm_moe_gb300 as bsg
    dev = "cuda"
    tokens, q_lora, heads = 256, 72, 2
    x = torch.zeros((tokens, q_lora), dtype=torch.bfloat16, device=dev)
    w = torch.zeros((heads * 192, q_lora), dtype=torch.bfloat16, device=dev)
    tab = torch.zeros((tokens, 64), dtype=torch.bfloat16, device=dev)
    o_row = torch.zeros((tokens, heads, 192), dtype=torch.uint8, device=dev)
    s_row = torch.zeros((tokens, heads, 6), dtype=torch.uint8, device=dev)
    o_col = torch.zeros((tokens, heads, 192), dtype=torch.uint8, device=dev)
    s_col = torch.zeros((tokens // 32, heads, 192), dtype=torch.uint8, device=dev)
    ws = torch.zeros(bsg.bsg_workspace_size(), dtype=torch.uint8, device=dev)

    def call(cta_pair=0, **kw):
        a = dict(tokens=tokens, q_lora=q_lora, heads=heads, hd=192, wsb=ws.numel())
        a.update(kw)
        o = bsg._opts(cta_pair=cta_pair)
        return bsg.raw_status("bsg_gemm_rope_bf16", x.data_ptr(), w.data_ptr(), tab.data_ptr(), tab.data_ptr(),
                              a["tokens"], a["q_lora"], a["heads"], a["hd"], 64, o_row.data_ptr(), s_row.data_ptr(),
                              o_col.data_ptr(), s_col.data_ptr(), ctypes.byref(o), ws.data_ptr(), a["wsb"], None)
    assert call(tokens=100) == 1 and call(q_lora=68) == 1
    assert call(hd=128) == 2 and call(cta_pair=2, tokens=128) == 1
    assert call(wsb=16) == 8
    assert call() == 0
    torch.cuda.synchronize()
    assert bsg.bsg_read_device_error(ws) == 0
    with pytest.raises(TypeError):
        from nvfp4_gemm_moe_gb300 import torch_ops
        torch_ops.gemm_rope_bf16(x.float(), w, tab, tab, heads)

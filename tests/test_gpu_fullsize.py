"""GPU parity at the full sizes of the named workloads, launched as bench.py launches them.

The outputs are too large for the oracle to recompute whole, so the checks are
* sampled outputs the oracle computes one by one: blocks of rows x columns spread over the
  batches or experts (first, last, ragged and empty ranges included), each checked with the
  same tolerance rules as the small parity tests;
* the sampled rows' operand codes and scale bytes, bit-exact against the oracle's quantiser;
* properties that hold at any size: the global amax equals max |C| of the whole GPU output up
  to C's own rounding, each expert's amax equals max |D| over that expert's rows, and empty
  experts give zero.
Inputs are the workloads' seeded recipes; nothing here depends on the CUDA path's values.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats, gemm as og, quantize as oq, sf_layout
from parity import TOL_C, check_c, check_d_bf16, check_e4m3_blocks, d_tolerance

pytestmark = pytest.mark.gpu


def _deq_rows(x_rows, fmt):
    """Oracle codes, logical scales and float64 dequantised values of fp32 rows (R, K)."""
    codes, sf_log = oq.quantize_logical(x_rows[None], fmt)
    v = 32 if fmt == "mxfp8" else 16
    vals = oq.decode_codes(codes[0], fmt)
    scales = oq.decode_scales(sf_log[0], fmt)
    return codes[0], sf_log[0], vals * np.repeat(scales, v, axis=-1)


def _check_operand_rows(q_gpu, sf_gpu, flat_rows, rows_per_batch, x_rows, fmt, k):
    """The GPU quantiser's codes and scale bytes of the sampled rows equal the oracle's."""
    codes, sf_log, deq = _deq_rows(x_rows, fmt)
    q = q_gpu.reshape(-1, q_gpu.shape[-1])
    got = q[torch.as_tensor(flat_rows, device=q.device)].cpu().numpy()
    assert np.array_equal(got, codes), "operand codes differ from the oracle's"
    v = 32 if fmt == "mxfp8" else 16
    sf = sf_layout.unpack_rows(sf_gpu.cpu().numpy(), flat_rows, k // v, rows_per_batch)
    assert np.array_equal(sf, sf_log), "operand scale bytes differ from the oracle's"
    return deq


@pytest.mark.parametrize("wl", [W.DENSE_MXFP8_8192, W.DENSE_NVFP4_16384], ids=lambda w: w.name)
def test_dense_full_size_sampled(lib, wl):
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg
    fmt, m, n, k, l = wl.fmt, wl.m, wl.n, wl.k, wl.l
    a = torch.from_numpy(wl.a_rows()).cuda()
    b = torch.from_numpy(wl.b_rows()).cuda()
    qa, sfa = torch_ops.quantize(a, fmt)
    qb, sfb = torch_ops.quantize(b, fmt)
    del a, b
    ws = torch_ops.new_workspace()
    c_dtype = torch.bfloat16 if wl.c_dtype == "bf16" else torch.float32
    c, amax = torch_ops.gemm_amax(qa, qb, sfa, sfb, fmt, m, n, k, l, c_dtype=c_dtype, workspace=ws)
    torch.cuda.synchronize()
    assert bsg.bsg_read_device_error(ws) == 0

    rng = np.random.default_rng(11)
    sampled_max = 0.0
    for batch in sorted({0, l - 1}):
        ms = np.unique(np.concatenate([[0, 127, 128, m - 1], rng.choice(m, 8, replace=False)]))
        ns = np.unique(np.concatenate([[0, 255, 256, n - 1], rng.choice(n, 8, replace=False)]))
        ra, rb = batch * m + ms, batch * n + ns
        ahat = _check_operand_rows(qa, sfa, ra, m, wl.a_rows(ra), fmt, k)
        bhat = _check_operand_rows(qb, sfb, rb, n, wl.b_rows(rb), fmt, k)
        ref = ahat @ bhat.T
        s = np.abs(ahat) @ np.abs(bhat).T
        got = c[batch][torch.as_tensor(ms).cuda()][:, torch.as_tensor(ns).cuda()].float().cpu().numpy()
        check_c(got, ref, s, wl.c_dtype, what=f"C[batch {batch}]")
        sampled_max = max(sampled_max, float(np.abs(ref).max()))

    # amax is of the fp32 accumulator; the stored C is that value rounded
    a_gpu = float(amax.cpu()[0])
    c_max = float(c.abs().max().float().cpu())
    ulp = float(formats.bf16_ulp(np.array([a_gpu]))[0]) if wl.c_dtype == "bf16" else 2.0 ** -23 * a_gpu
    assert abs(a_gpu - c_max) <= ulp, (a_gpu, c_max)
    assert a_gpu >= sampled_max * (1 - 1e-5)


def _grouped_inputs(wl):
    from nvfp4_gemm_moe_gb300 import torch_ops
    offs = wl.padded_offsets()
    a = torch.from_numpy(wl.a_rows()).cuda()
    qa, sfa = torch_ops.quantize(a[None], wl.fmt)
    del a
    b = torch.from_numpy(wl.b_rows()).cuda()
    qb, sfb = torch_ops.quantize(b, wl.fmt)
    del b
    return offs, qa, sfa, qb, sfb


def _sample_blocks(wl, offs, rng):
    """32-row x 32-column blocks: in the largest, a small and the last non-empty expert, in a
    padding range and at the first and last columns."""
    ends = np.asarray(offs, dtype=np.int64)
    begins = np.concatenate([[0], ends[:-1]])
    sizes = ends - begins
    nonempty = np.flatnonzero(sizes > 0)
    counts = wl.counts()
    picks = {int(nonempty[np.argmax(sizes[nonempty])]), int(nonempty[np.argmin(sizes[nonempty])]), int(nonempty[-1])}
    blocks = []
    for g in sorted(picks):
        r_first = int(begins[g])
        r_pad = int(begins[g] + counts[g]) // 32 * 32  # the block holding the last routed rows / padding
        for r0 in sorted({r_first, min(r_pad, int(ends[g]) - 32)}):
            for c0 in sorted({0, wl.n - 32, int(rng.integers(0, wl.n // 32)) * 32}):
                blocks.append((g, r0, c0))
    return blocks


@pytest.mark.parametrize("wl", [W.GROUPED_SRELU_E32, W.GROUPED_SRELU_E32_CLAMP, W.GROUPED_FP8D_E128],
                         ids=lambda w: w.name)
def test_grouped_full_size_sampled(lib, wl):
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg
    n, k, fmt = wl.n, wl.k, wl.fmt
    offs, qa, sfa, qb, sfb = _grouped_inputs(wl)
    vm = int(offs[-1])
    alpha, prob = wl.alpha(), wl.prob()
    nc = 1.0
    ws = torch_ops.new_workspace()
    out = torch_ops.grouped_gemm_srelu(
        qa[0], qb, sfa, sfb, fmt, torch.from_numpy(offs).cuda(), torch.from_numpy(alpha).cuda(),
        torch.from_numpy(prob).cuda(), n, k, tanh_clamp_scale=wl.tanh_clamp, d_dtype=wl.d_dtype,
        norm_const=torch.tensor([nc], dtype=torch.float32, device="cuda"), workspace=ws)
    torch.cuda.synchronize()
    assert bsg.bsg_read_device_error(ws) == 0

    rng = np.random.default_rng(5)
    for g, r0, c0 in _sample_blocks(wl, offs, rng):
        rows = np.arange(r0, r0 + 32)
        cols = np.arange(c0, c0 + 32)
        ahat = _check_operand_rows(qa, sfa, rows, vm, wl.a_rows(rows), fmt, k)
        bhat = _check_operand_rows(qb, sfb, g * n + cols, n, wl.b_rows(g * n + cols), fmt, k)
        c_ref = float(alpha[g]) * (ahat @ bhat.T)
        s = float(alpha[g]) * (np.abs(ahat) @ np.abs(bhat).T)
        c_tol = TOL_C * s
        d_ref = og.srelu(c_ref, prob[rows], wl.tanh_clamp)
        rt, ct = torch.as_tensor(rows).cuda(), torch.as_tensor(cols).cuda()
        check_c(out["c"][rt][:, ct].float().cpu().numpy(), c_ref, s, "bf16", what=f"C[e{g}, {r0}, {c0}]")
        if wl.d_dtype == "bf16":
            check_d_bf16(out["d"][rt][:, ct].float().cpu().numpy(), d_ref, c_ref, prob[rows], c_tol,
                         what=f"D[e{g}, {r0}, {c0}]")
        else:
            d_tol = d_tolerance(c_ref, prob[rows], c_tol) + 2.0 ** -20 * d_ref
            sf_row = sf_layout.unpack_rows(out["sfd_row"].cpu().numpy(), rows, n // 32, vm)[:, c0 // 32:c0 // 32 + 1]
            sf_col = sf_layout.unpack_rows(out["sfd_col"].cpu().numpy(), cols, vm // 32, n)[:, r0 // 32:r0 // 32 + 1]
            check_e4m3_blocks(out["d"][rt][:, ct].cpu().numpy(), sf_row, d_ref, d_tol, nc, axis=1, what="D_row")
            check_e4m3_blocks(out["d_col"][rt][:, ct].cpu().numpy(), sf_col, d_ref, d_tol, nc, axis=0, what="D_col")

    if wl.d_dtype == "bf16":
        # each expert's amax is max |D| of its rows (fp32, before D's own rounding); empty ones are 0
        amax = out["amax"].cpu().numpy()
        begin = 0
        for g, end in enumerate(offs):
            end = int(end)
            if end == begin:
                assert amax[g] == 0.0
            else:
                d_max = float(out["d"][begin:end].float().abs().max().cpu())
                assert abs(amax[g] - d_max) <= float(formats.bf16_ulp(np.array([amax[g]]))[0]), (g, amax[g], d_max)
            begin = end


def test_rope_full_size_sampled(lib):
    """The 16384-token DeepSeek-V3 Q up-projection: 32-token blocks x single heads recomputed by
    the oracle (row and column scales of a block depend only on its own 32 tokens / features)."""
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg
    from oracle import rope as orope
    from test_gpu_rope import _tolerance
    wl = W.ROPE_PROJ_T16384
    x = torch.from_numpy(wl.x_rows()).cuda()
    w = torch.from_numpy(wl.w_rows()).cuda()
    qx, sx = torch_ops.quantize(x, "mxfp8")
    qw, sw = torch_ops.quantize(w, "mxfp8")
    del x, w
    cos32, sin32 = wl.tables()
    cos = torch.from_numpy(cos32).to(torch.bfloat16)
    sin = torch.from_numpy(sin32).to(torch.bfloat16)
    ws = torch_ops.new_workspace()
    out = torch_ops.gemm_rope_mxfp8(qx[0], sx, qw[0], sw, cos.cuda(), sin.cuda(), wl.heads, wl.head_dim, wl.qk_rope,
                                    workspace=ws)
    torch.cuda.synchronize()
    assert bsg.bsg_read_device_error(ws) == 0
    d = wl.head_dim
    for t0 in (0, 8192, wl.tokens - 32):
        rows = np.arange(t0, t0 + 32)
        xc, xs = oq.quantize_logical(wl.x_rows(rows)[None], "mxfp8")
        assert np.array_equal(qx[0][t0:t0 + 32].cpu().numpy(), xc[0])
        for h in (0, 77, wl.heads - 1):
            wrows = np.arange(h * d, (h + 1) * d)
            wc, wsc = oq.quantize_logical(wl.w_rows(wrows)[None], "mxfp8")
            c64 = cos[t0:t0 + 32].double().numpy()
            s64 = sin[t0:t0 + 32].double().numpy()
            ref = orope.project(xc[0], xs[0], wc[0], wsc[0], c64, s64, 1, d, wl.qk_rope)
            xh, wh = orope.dequantize_plain(xc[0], xs[0]), orope.dequantize_plain(wc[0], wsc[0])
            tol = _tolerance((xh @ wh.T).reshape(32, 1, d), (np.abs(xh) @ np.abs(wh).T).reshape(32, 1, d), c64, s64,
                             d, wl.qk_rope).reshape(32, d)
            y = ref["y"].reshape(32, d)
            check_e4m3_blocks(out["out_fp8_row"][t0:t0 + 32, h].cpu().numpy(),
                              out["out_scales_row"][t0:t0 + 32, h].cpu().numpy(), y, tol, 1.0, axis=1,
                              what=f"row[t{t0}, h{h}]")
            check_e4m3_blocks(out["out_fp8_col"][t0:t0 + 32, h].cpu().numpy(),
                              out["out_scales_col"][t0 // 32, h].cpu().numpy()[:, None], y, tol, 1.0, axis=0,
                              what=f"col[t{t0}, h{h}]")


def test_rope_bf16_full_size_sampled(lib):
    """The same projection with bf16 operands: 32-token blocks x single heads recomputed by the
    oracle from the bf16 values."""
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg
    from oracle import rope as orope
    from test_gpu_rope import _tolerance
    wl = W.ROPE_PROJ_BF16_T16384
    x = torch.from_numpy(wl.x_rows()).to(torch.bfloat16)
    w = torch.from_numpy(wl.w_rows()).to(torch.bfloat16)
    cos32, sin32 = wl.tables()
    cos = torch.from_numpy(cos32).to(torch.bfloat16)
    sin = torch.from_numpy(sin32).to(torch.bfloat16)
    ws = torch_ops.new_workspace()
    out = torch_ops.gemm_rope_bf16(x.cuda(), w.cuda(), cos.cuda(), sin.cuda(), wl.heads, wl.head_dim, wl.qk_rope,
                                   workspace=ws)
    torch.cuda.synchronize()
    assert bsg.bsg_read_device_error(ws) == 0
    d = wl.head_dim
    for t0 in (0, 8192, wl.tokens - 32):
        xh = x[t0:t0 + 32].double().numpy()
        for h in (0, 77, wl.heads - 1):
            wh = w[h * d:(h + 1) * d].double().numpy()
            c64 = cos[t0:t0 + 32].double().numpy()
            s64 = sin[t0:t0 + 32].double().numpy()
            ref = orope.project_bf16(xh, wh, c64, s64, 1, d, wl.qk_rope)
            tol = _tolerance((xh @ wh.T).reshape(32, 1, d), (np.abs(xh) @ np.abs(wh).T).reshape(32, 1, d), c64, s64,
                             d, wl.qk_rope).reshape(32, d)
            y = ref["y"].reshape(32, d)
            check_e4m3_blocks(out["out_fp8_row"][t0:t0 + 32, h].cpu().numpy(),
                              out["out_scales_row"][t0:t0 + 32, h].cpu().numpy(), y, tol, 1.0, axis=1,
                              what=f"row[t{t0}, h{h}]")
            check_e4m3_blocks(out["out_fp8_col"][t0:t0 + 32, h].cpu().numpy(),
                              out["out_scales_col"][t0 // 32, h].cpu().numpy()[:, None], y, tol, 1.0, axis=0,
                              what=f"col[t{t0}, h{h}]")


def test_dswiglu_full_size_sampled(lib):
    """The E32 dSwiGLU backward at full size: 32-row blocks (largest, smallest and last
    expert) recomputed by the oracle over all 2N columns of D and their dprob rows."""
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg
    from oracle import dswiglu as od
    from parity import check_float_out, dprob_tolerance, dswiglu_tolerances
    wl = W.GROUPED_DSWIGLU_E32
    n, k, fmt = wl.n, wl.k, wl.fmt
    offs, qa, sfa, qb, sfb = _grouped_inputs(wl)
    vm = int(offs[-1])
    alpha, beta, prob = wl.alpha(), wl.beta(), wl.prob()
    c = torch.from_numpy(wl.c_rows()).to(torch.bfloat16)
    ws = torch_ops.new_workspace()
    out = torch_ops.grouped_gemm_dswiglu(qa[0], qb, sfa, sfb, fmt, torch.from_numpy(offs).cuda(),
                                         torch.from_numpy(alpha).cuda(), torch.from_numpy(beta).cuda(),
                                         torch.from_numpy(prob).cuda(), c.cuda(), n, k, workspace=ws)
    torch.cuda.synchronize()
    assert bsg.bsg_read_device_error(ws) == 0
    ends = np.asarray(offs, dtype=np.int64)
    begins = np.concatenate([[0], ends[:-1]])
    sizes = ends - begins
    nonempty = np.flatnonzero(sizes > 0)
    for g in sorted({int(nonempty[np.argmax(sizes[nonempty])]), int(nonempty[np.argmin(sizes[nonempty])]),
                     int(nonempty[-1])}):
        r0 = int(begins[g])
        rows = np.arange(r0, r0 + 32)
        ahat = _check_operand_rows(qa, sfa, rows, vm, wl.a_rows(rows), fmt, k)
        bhat = _check_operand_rows(qb, sfb, g * n + np.arange(n), n, wl.b_rows(g * n + np.arange(n)), fmt, k)
        ref = float(alpha[g]) * (ahat @ bhat.T)
        ref_tol = TOL_C * float(alpha[g]) * (np.abs(ahat) @ np.abs(bhat).T)
        cv = c[r0:r0 + 32].double().numpy() * float(beta[g])
        x, gate = od.deinterleave(cv)
        ab, dsw, dprob = od.epilogue(ref, x, gate, prob[rows])
        r = {"ref": ref, "x": x, "gate": gate, "ab": ab, "dswiglu": dsw}
        t_ab, t_dsw = dswiglu_tolerances(r, ref_tol, prob[rows])
        check_float_out(out["d_row"][r0:r0 + 32].float().cpu().numpy(), od.interleave(ab, dsw),
                        od.interleave(t_ab, t_dsw), "bf16", what=f"D[e{g}, rows {r0}..]")
        dp = out["dprob"][r0:r0 + 32].cpu().numpy().astype(np.float64)
        assert np.all(np.abs(dp - dprob) <= dprob_tolerance(r, ref_tol, 128, 2 * (n // 128) + 2)), (g, dp, dprob)

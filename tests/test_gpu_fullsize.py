"""GPU parity at the full sizes of the named workloads, launched as bench.py launches them.

* The dense workloads (L = 4 MXFP8 8192^3, NVFP4 16384 x 16384 x 8192) and the grouped ones
  (32 experts with bf16 D, without and with the tanh clamp; 128 Zipf-routed experts with E4M3 D
  and its row and column scales) are compared with the oracle element by element: every
  operand code and scale byte, every element of C and D (D_col, SFD_row, SFD_col), the global
  amax and each expert's amax.  The oracle runs on row bands and experts in turn (host memory
  stays bounded) with its quantiser split over host threads (``fullsize``).
* The RoPE projection and the dSwiGLU backward are checked on sampled blocks the oracle
  computes one by one, with the same tolerance rules as the small parity tests.
Inputs are the workloads' seeded recipes; nothing here depends on the CUDA path's values.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats, gemm as og, quantize as oq, sf_layout
import fullsize
from parity import TOL_C, check_amax, check_c, check_d_bf16, check_e4m3_blocks, d_tolerance

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


DENSE_BAND = 2048  # rows of A per oracle band (bounds the host memory of the float64 products)


@pytest.mark.parametrize("wl", [W.DENSE_MXFP8_8192, W.DENSE_NVFP4_16384], ids=lambda w: w.name)
def test_dense_full_size_elementwise(lib, wl):
    """Every element of C of the large dense workloads against the oracle ("GEMM + Amax (SM100)",
    Equations), in bands of rows per batch; every operand code and scale byte bit-exact; the
    global amax against the oracle's max |C|."""
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
    sfa_h, sfb_h = sfa.cpu().numpy(), sfb.cpu().numpy()
    qa2, qb2 = qa.reshape(l * m, -1), qb.reshape(l * n, -1)

    ref_max, checked = 0.0, 0
    for batch in range(l):
        bhat = fullsize.checked_operand(wl.b_rows, batch * n, (batch + 1) * n,
                                        qb2[batch * n:(batch + 1) * n].cpu().numpy(), sfb_h, n, fmt, k, "B")
        babs_t = np.abs(bhat).T
        bhat_t = bhat.T
        for r0 in range(0, m, DENSE_BAND):
            r1 = min(r0 + DENSE_BAND, m)
            ahat = fullsize.checked_operand(wl.a_rows, batch * m + r0, batch * m + r1,
                                            qa2[batch * m + r0:batch * m + r1].cpu().numpy(), sfa_h, m, fmt, k, "A")
            ref = ahat @ bhat_t
            s = np.abs(ahat) @ babs_t
            got = c[batch, r0:r1].float().cpu().numpy()
            fullsize.run_checks(lambda i, j: check_c(got[i:j], ref[i:j], s[i:j], wl.c_dtype,
                                                     what=f"C[batch {batch}, rows {r0 + i}..{r0 + j - 1}]"), r1 - r0)
            ref_max = max(ref_max, float(np.abs(ref).max()))
            checked += ref.size
    assert checked == l * m * n
    check_amax(np.array([float(amax.cpu()[0])]), np.array([ref_max]), what="global amax")


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


def _bf16_beyond_ulp(d_gpu, d_ref):
    """Elements whose bf16 D is more than one bf16 ulp from the oracle (inside the tolerance only
    through the carried C term)."""
    return int(np.count_nonzero(np.abs(d_gpu - d_ref) > formats.bf16_ulp(d_ref)))


def test_grouped_bf16_full_size_elementwise(lib):
    """The 32-expert sReLU workload, without and with the tanh clamp (s = 32): every element of C
    and D of every expert against the oracle ("Grouped GEMM + sReLU (SM100)", Equations and Tanh
    soft clamp), every operand code and scale byte, and each expert's amax."""
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg
    wl, wl_c = W.GROUPED_SRELU_E32, W.GROUPED_SRELU_E32_CLAMP
    n, k, fmt = wl.n, wl.k, wl.fmt
    offs, qa, sfa, qb, sfb = _grouped_inputs(wl)
    vm = int(offs[-1])
    alpha, prob = wl.alpha(), wl.prob()
    ws = torch_ops.new_workspace()
    args = (qa[0], qb, sfa, sfb, fmt, torch.from_numpy(offs).cuda(), torch.from_numpy(alpha).cuda(),
            torch.from_numpy(prob).cuda(), n, k)
    outs = [torch_ops.grouped_gemm_srelu(*args, tanh_clamp_scale=w.tanh_clamp, d_dtype="bf16", workspace=ws)
            for w in (wl, wl_c)]
    torch.cuda.synchronize()
    assert bsg.bsg_read_device_error(ws) == 0
    sfa_h, sfb_h = sfa.cpu().numpy(), sfb.cpu().numpy()
    qa2, qb2 = qa[0], qb.reshape(wl.experts * n, -1)
    amax_ref = np.zeros((2, wl.experts))
    beyond = [0, 0]
    begin = 0
    for g, end in enumerate(offs):
        end = int(end)
        if end == begin:
            continue
        bhat = fullsize.checked_operand(wl.b_rows, g * n, (g + 1) * n, qb2[g * n:(g + 1) * n].cpu().numpy(), sfb_h,
                                        n, fmt, k, f"B[e{g}]")
        ahat = fullsize.checked_operand(wl.a_rows, begin, end, qa2[begin:end].cpu().numpy(), sfa_h, vm, fmt, k,
                                        f"A[e{g}]")
        c_ref = float(alpha[g]) * (ahat @ bhat.T)
        s = float(alpha[g]) * (np.abs(ahat) @ np.abs(bhat).T)
        p = prob[begin:end]
        for i, (w, out) in enumerate(zip((wl, wl_c), outs)):
            d_ref = og.srelu(c_ref, p, w.tanh_clamp)
            c_got = out["c"][begin:end].float().cpu().numpy()
            d_got = out["d"][begin:end].float().cpu().numpy()

            def check(a, b, c_got=c_got, d_got=d_got, d_ref=d_ref):
                check_c(c_got[a:b], c_ref[a:b], s[a:b], "bf16", what=f"C[e{g}, rows {begin + a}..]")
                check_d_bf16(d_got[a:b], d_ref[a:b], c_ref[a:b], p[a:b], TOL_C * s[a:b],
                             what=f"D[{w.name}, e{g}, rows {begin + a}..]")
                return _bf16_beyond_ulp(d_got[a:b], d_ref[a:b])
            beyond[i] += sum(fullsize.run_checks(check, end - begin))
            amax_ref[i, g] = np.abs(d_ref).max()
        begin = end
    for i, out in enumerate(outs):
        got = out["amax"].cpu().numpy().astype(np.float64)
        empty = amax_ref[i] == 0
        assert np.all(got[empty] == 0)
        check_amax(got[~empty], amax_ref[i][~empty], what="per-expert amax")
    print(f"bf16 D elements beyond one ulp of the oracle (inside the carried C bound): "
          f"{beyond[0]} (no clamp), {beyond[1]} (tanh clamp) of {vm * n} each")


def test_grouped_fp8d_full_size_elementwise(lib):
    """The 128-expert Zipf-routed workload with E4M3 D: every element of C, D and D_col and every
    SFD_row / SFD_col byte of every expert against the oracle ("Grouped GEMM + sReLU (SM100)",
    Equations and Shapes), every operand code and scale byte; the run with C = NULL gives the
    same D, D_col and scale bytes."""
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg
    wl = W.GROUPED_FP8D_E128
    n, k, fmt = wl.n, wl.k, wl.fmt
    offs, qa, sfa, qb, sfb = _grouped_inputs(wl)
    vm = int(offs[-1])
    alpha, prob = wl.alpha(), wl.prob()
    nc = 1.0
    ws = torch_ops.new_workspace()
    args = (qa[0], qb, sfa, sfb, fmt, torch.from_numpy(offs).cuda(), torch.from_numpy(alpha).cuda(),
            torch.from_numpy(prob).cuda(), n, k)
    ncd = torch.tensor([nc], dtype=torch.float32, device="cuda")
    out = torch_ops.grouped_gemm_srelu(*args, d_dtype="e4m3", norm_const=ncd, workspace=ws)
    out0 = torch_ops.grouped_gemm_srelu(*args, d_dtype="e4m3", norm_const=ncd, c_dtype=None, workspace=ws)
    torch.cuda.synchronize()
    assert bsg.bsg_read_device_error(ws) == 0
    for key in ("d", "d_col", "sfd_row", "sfd_col"):
        assert torch.equal(out[key], out0[key]), key
    del out0
    sfa_h, sfb_h = sfa.cpu().numpy(), sfb.cpu().numpy()
    qa2, qb2 = qa[0], qb.reshape(wl.experts * n, -1)
    sfd_row_h = out["sfd_row"].cpu().numpy()
    sf_col = sf_layout.unpack(out["sfd_col"].cpu().numpy(), n, vm // 32)[0]  # (N, valid_m / 32)
    begin = 0
    for g, end in enumerate(offs):
        end = int(end)
        if end == begin:
            continue
        bhat = fullsize.checked_operand(wl.b_rows, g * n, (g + 1) * n, qb2[g * n:(g + 1) * n].cpu().numpy(), sfb_h,
                                        n, fmt, k, f"B[e{g}]")
        ahat = fullsize.checked_operand(wl.a_rows, begin, end, qa2[begin:end].cpu().numpy(), sfa_h, vm, fmt, k,
                                        f"A[e{g}]")
        c_ref = float(alpha[g]) * (ahat @ bhat.T)
        s = float(alpha[g]) * (np.abs(ahat) @ np.abs(bhat).T)
        p = prob[begin:end]
        d_ref = og.srelu(c_ref, p)
        d_tol = d_tolerance(c_ref, p, TOL_C * s) + 2.0 ** -20 * d_ref
        c_got = out["c"][begin:end].float().cpu().numpy()
        d_got = out["d"][begin:end].cpu().numpy()
        dc_got = out["d_col"][begin:end].cpu().numpy()
        sf_row = sf_layout.unpack_rows(sfd_row_h, np.arange(begin, end), n // 32, vm)

        def check(a, b):
            # a, b: 32-row aligned (the chunks are 256 rows), so column blocks lie inside a chunk
            check_c(c_got[a:b], c_ref[a:b], s[a:b], "bf16", what=f"C[e{g}, rows {begin + a}..]")
            check_e4m3_blocks(d_got[a:b], sf_row[a:b], d_ref[a:b], d_tol[a:b], nc, axis=1,
                              what=f"D_row[e{g}, rows {begin + a}..]")
            check_e4m3_blocks(dc_got[a:b], sf_col[:, (begin + a) // 32:(begin + b) // 32], d_ref[a:b], d_tol[a:b],
                              nc, axis=0, what=f"D_col[e{g}, rows {begin + a}..]")
        fullsize.run_checks(check, end - begin)
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

"""GPU parity of bsg_grouped_gemm_dswiglu (grouped GEMM + dSwiGLU backward) against the oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import dswiglu as od, formats, quantize as oq, sf_layout
from guards import Outputs
from parity import TOL_C, check_e4m3_blocks, check_float_out, dprob_tolerance, dswiglu_tolerances

pytestmark = pytest.mark.gpu

EDGE = [0, 300, 0, 0, 1, 256, 0]  # empty experts first, in a run and last; one 1-row expert


def _c_input(wl, c_kind, seed):
    """The stored forward intermediate as a device tensor and its exact values (float64)."""
    if c_kind == "e4m3":
        rng = np.random.default_rng(seed)
        codes = rng.integers(0, 256, size=(wl.valid_m, 2 * wl.n), dtype=np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0x00  # no NaN codes
        return torch.from_numpy(codes).cuda(), formats.decode_e4m3(codes)
    c = torch.from_numpy(wl.c_rows())
    c = c.to({"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[c_kind])
    return c.cuda(), c.double().numpy()


def run_dswiglu(counts, n, k, d_dtype="bf16", c_kind="bf16", fmt="mxfp8", tile_n=0, cta_pair=0, nc=1.0,
                max_ctas=0, seed=5):
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg
    wl = W.GroupedDswiglu("t", len(counts), k, n, int(sum(counts)), "fixed:" + ",".join(str(c) for c in counts),
                          d_dtype, seed=seed, fmt=fmt)
    offs = wl.padded_offsets()
    vm = int(offs[-1])
    a, b = wl.a_rows(), wl.b_rows()
    alpha, beta, prob = wl.alpha(), wl.beta(), wl.prob()
    c_dev, c_vals = _c_input(wl, c_kind, seed)
    qa, sfa = torch_ops.quantize(torch.from_numpy(a).cuda(), fmt)
    qb, sfb = torch_ops.quantize(torch.from_numpy(b).cuda(), fmt)
    ws = torch_ops.new_workspace()
    g = Outputs()
    outputs = {"dprob": g.zeros("dprob", (vm,))}
    if d_dtype == "e4m3":
        outputs.update(d_row=g.codes("d_row", (vm, 2 * n)), d_col=g.codes("d_col", (vm, 2 * n)),
                       sfd_row=g.scales("sfd_row", bsg.bsg_sf_bytes(1, vm, 2 * n, 32)),
                       sfd_col=g.scales("sfd_col", bsg.bsg_sf_bytes(1, 2 * n, vm, 32)))
    else:
        outputs.update(d_row=g.float("d_row", (vm, 2 * n), {"bf16": torch.bfloat16, "f16": torch.float16,
                                                            "f32": torch.float32}[d_dtype]),
                       amax=g.float("amax", (len(counts), 2), torch.float32))
    out = torch_ops.grouped_gemm_dswiglu(
        qa[0], qb, sfa, sfb, fmt, torch.from_numpy(offs).cuda(), torch.from_numpy(alpha).cuda(),
        torch.from_numpy(beta).cuda(), torch.from_numpy(prob).cuda(), c_dev, n, k,
        c_dtype="e4m3" if c_kind == "e4m3" else None, d_dtype=d_dtype,
        norm_const=torch.tensor([nc], dtype=torch.float32, device="cuda"), workspace=ws, tile_n=tile_n,
        cta_pair=cta_pair, max_ctas=max_ctas, outputs=outputs)
    torch.cuda.synchronize()
    g.check()
    assert bsg.bsg_read_device_error(ws) == 0

    qa_ref, sfa_ref = oq.quantize(a, fmt)
    qb_ref, sfb_ref = oq.quantize(b, fmt)
    assert np.array_equal(qa.cpu().numpy(), qa_ref) and np.array_equal(qb.cpu().numpy(), qb_ref)
    assert np.array_equal(sfa.cpu().numpy(), sfa_ref) and np.array_equal(sfb.cpu().numpy(), sfb_ref)
    ref = od.grouped_dswiglu(qa_ref[0], qb_ref, sfa_ref, sfb_ref, fmt, offs, alpha, beta, prob, c_vals, k, n,
                             d_fp8=(d_dtype == "e4m3"), norm_const=nc)
    # ref bound: 2^-20 * alpha_g * sum_k |Ahat||Bhat| per element
    ahat = np.abs(oq.dequantize(qa_ref, sfa_ref, fmt, vm, k, 1)[0])
    bhat = np.abs(oq.dequantize(qb_ref, sfb_ref, fmt, n, k, len(counts)))
    g_of = np.maximum(od.gemm.expert_of_rows(offs, vm), 0)
    s = np.zeros((vm, n))
    for g in range(len(counts)):
        rows = g_of == g
        if rows.any():
            s[rows] = float(alpha[g]) * (ahat[rows] @ bhat[g].T)
    ref_tol = TOL_C * s
    tol_ab, tol_dsw = dswiglu_tolerances(ref, ref_tol, prob)
    tol_d = od.interleave(tol_ab, tol_dsw)

    dprob = out["dprob"].cpu().numpy().astype(np.float64)
    dp_tol = dprob_tolerance(ref, ref_tol, 128, 2 * (-(-n // 128)) + 2)
    bad = ~(np.abs(dprob - ref["dprob"]) <= dp_tol)
    assert not bad.any(), (np.flatnonzero(bad)[:5], dprob[bad][:5], ref["dprob"][bad][:5])

    if d_dtype in ("bf16", "f16", "f32"):
        d_gpu = out["d_row"].float().cpu().numpy()
        check_float_out(d_gpu, ref["d"], tol_d, d_dtype, what="D")
        amax = out["amax"].cpu().numpy().astype(np.float64)
        assert amax.shape == (len(counts), 2)
        begin = 0
        for g, end in enumerate(offs):
            end = int(end)
            if end == begin:
                assert np.all(amax[g] == 0.0), (g, amax[g])
            else:
                for j, t in ((0, tol_ab), (1, tol_dsw)):
                    bound = t[begin:end].max() * (1 + 1e-9) + 1e-30
                    assert abs(amax[g, j] - ref["amax"][g, j]) <= bound, (g, j, amax[g, j], ref["amax"][g, j])
            begin = end
        return out, ref
    sfd_row = sf_layout.unpack(out["sfd_row"].cpu().numpy(), vm, 2 * n // 32)[0]
    sfd_col = sf_layout.unpack(out["sfd_col"].cpu().numpy(), 2 * n, vm // 32)[0]
    check_e4m3_blocks(out["d_row"].cpu().numpy(), sfd_row, ref["d"], tol_d, nc, axis=1, what="D_row")
    check_e4m3_blocks(out["d_col"].cpu().numpy(), sfd_col, ref["d"], tol_d, nc, axis=0, what="D_col")
    # padding bytes of the SF buffers are zero
    assert np.array_equal(sf_layout.pack(sfd_row[None]), out["sfd_row"].cpu().numpy())
    assert np.array_equal(sf_layout.pack(sfd_col[None]), out["sfd_col"].cpu().numpy())
    return out, ref


@pytest.mark.parametrize("n,k,tile_n,cta_pair", [
    (256, 512, 0, 0),
    (256, 512, 256, 1),
    (288, 512, 256, 1),     # ragged second tile (one 32-column chunk)
    (448, 384, 224, 1),     # 224-wide tiles starting inside a 128-row scale atom
    (96, 256, 128, 1),      # N below one tile; 2N not a multiple of 128
    (512, 512, 0, 2),       # CTA pairs
    (448, 512, 224, 2),
])
def test_dswiglu_bf16(lib, n, k, tile_n, cta_pair):
    run_dswiglu(EDGE, n, k, "bf16", "bf16", tile_n=tile_n, cta_pair=cta_pair)


@pytest.mark.parametrize("c_kind,d_dtype,cta_pair", [
    ("f16", "f16", 1), ("f32", "f32", 2), ("e4m3", "bf16", 1), ("bf16", "f32", 1),
])
def test_dswiglu_c_and_d_types(lib, c_kind, d_dtype, cta_pair):
    run_dswiglu([300, 500, 0, 220], 256, 512, d_dtype, c_kind, cta_pair=cta_pair)


@pytest.mark.parametrize("nc,tile_n,cta_pair,n", [
    (1.0, 0, 0, 256), (0.75, 128, 1, 256), (1.0, 224, 1, 448), (1.0, 224, 2, 448), (0.5, 256, 2, 96),
])
def test_dswiglu_fp8_d(lib, nc, tile_n, cta_pair, n):
    run_dswiglu(EDGE, n, 512, "e4m3", "bf16", tile_n=tile_n, cta_pair=cta_pair, nc=nc)


@pytest.mark.parametrize("d_dtype,tile_n,cta_pair", [("bf16", 0, 0), ("f32", 128, 1), ("bf16", 256, 2)])
def test_dswiglu_nvfp4(lib, d_dtype, tile_n, cta_pair):
    run_dswiglu([1, 2, 3, 700, 4], 256, 1024, d_dtype, "bf16", fmt="nvfp4", tile_n=tile_n, cta_pair=cta_pair)


def test_dswiglu_few_ctas(lib):
    run_dswiglu([600, 900, 0, 300], 512, 512, "bf16", "bf16", tile_n=256, cta_pair=1, max_ctas=3)
    run_dswiglu([600, 900, 0, 300], 512, 512, "e4m3", "bf16", cta_pair=2, max_ctas=4)


def test_dswiglu_dprob_accumulates(lib):
    """dprob is added into: a second call on the same buffer doubles it (up to rounding)."""
    from nvfp4_gemm_moe_gb300 import torch_ops
    wl = W.GroupedDswiglu("t", 2, 256, 128, 400, "fixed:200,200", "bf16", seed=9)
    offs = torch.from_numpy(wl.padded_offsets()).cuda()
    qa, sfa = torch_ops.quantize(torch.from_numpy(wl.a_rows()).cuda(), "mxfp8")
    qb, sfb = torch_ops.quantize(torch.from_numpy(wl.b_rows()).cuda(), "mxfp8")
    c = torch.from_numpy(wl.c_rows()).to(torch.bfloat16).cuda()
    args = (qa[0], qb, sfa, sfb, "mxfp8", offs, torch.from_numpy(wl.alpha()).cuda(), torch.from_numpy(wl.beta()).cuda(),
            torch.from_numpy(wl.prob()).cuda(), c, 128, 256)
    out = torch_ops.grouped_gemm_dswiglu(*args)
    once = out["dprob"].clone()
    torch_ops.grouped_gemm_dswiglu(*args, outputs=out)
    torch.cuda.synchronize()
    assert torch.any(once != 0)
    torch.testing.assert_close(out["dprob"], 2 * once, rtol=1e-5, atol=1e-6)


def test_dswiglu_bad_offsets_detected_on_device(lib):
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg
    k, n, vm = 256, 128, 512
    qa = torch.zeros((vm, k), dtype=torch.uint8, device="cuda")
    qb = torch.zeros((2, n, k), dtype=torch.uint8, device="cuda")
    sfa = torch.zeros(bsg.bsg_sf_bytes(1, vm, k, 32), dtype=torch.uint8, device="cuda")
    sfb = torch.zeros(bsg.bsg_sf_bytes(2, n, k, 32), dtype=torch.uint8, device="cuda")
    c = torch.zeros((vm, 2 * n), dtype=torch.bfloat16, device="cuda")
    ws = torch_ops.new_workspace()
    offs = torch.tensor([100, 512], dtype=torch.int32, device="cuda")
    ones = torch.ones(2, device="cuda")
    prob = torch.ones(vm, device="cuda")
    torch_ops.grouped_gemm_dswiglu(qa, qb, sfa, sfb, "mxfp8", offs, ones, ones, prob, c, n, k, workspace=ws)
    assert bsg.bsg_read_device_error(ws) == bsg.DEVERR_BAD_OFFSETS


def test_dswiglu_max_experts(lib):
    """512 experts (the dSwiGLU limit: 2 x 512 amax values staged in shared memory)."""
    counts = [0] * 512
    counts[0], counts[300], counts[511] = 100, 256, 1
    run_dswiglu(counts, 128, 256, "bf16", "bf16")

"""GPU parity of bsg_grouped_gemm_srelu (grouped MoE GEMM + prob-gated sReLU) against the oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats, gemm as og, quantize as oq, sf_layout
from guards import Outputs
from parity import TOL_C, check_amax, check_c_float, check_d_float, check_e4m3_blocks, d_tolerance

pytestmark = pytest.mark.gpu


def _case(counts, n, k, seed=3, a_scale=1.0):
    wl = W.Grouped("t", len(counts), k, n, int(sum(counts)), "fixed:" + ",".join(str(c) for c in counts), "bf16",
                   seed=seed)
    offs = wl.padded_offsets()
    a = wl.a_rows() * np.float32(a_scale)
    b = wl.b_rows()
    return wl, offs, a.astype(np.float32), b, wl.alpha(), wl.prob()


def run_grouped(counts, n, k, d_dtype="bf16", clamp=None, c_kind="bf16", nc=1.0, tile_n=0, seed=3, a_scale=1.0,
                tanh_approx=False, max_ctas=0, cta_pair=0, fmt="mxfp8", discrete=False, b_major="k"):
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg
    wl, offs, a, b, alpha, prob = _case(counts, n, k, seed, a_scale)
    vm = int(offs[-1])
    qa, sfa = torch_ops.quantize(torch.from_numpy(a).cuda(), fmt)
    qb, sfb = torch_ops.quantize(torch.from_numpy(b).cuda(), fmt)
    ws = torch_ops.new_workspace()
    c_dtype = {"bf16": torch.bfloat16, "f32": torch.float32, "f16": torch.float16, None: None}[c_kind]
    g = Outputs()
    outputs = {"c": None if c_dtype is None else g.float("c", (vm, n), c_dtype)}
    if d_dtype == "e4m3":
        outputs.update(d=g.codes("d", (vm, n)), d_col=g.codes("d_col", (vm, n)),
                       sfd_row=g.scales("sfd_row", bsg.bsg_sf_bytes(1, vm, n, 32)),
                       sfd_col=g.scales("sfd_col", bsg.bsg_sf_bytes(1, n, vm, 32)))
    else:
        outputs.update(d=g.float("d", (vm, n), {"bf16": torch.bfloat16, "f16": torch.float16,
                                                "f32": torch.float32}[d_dtype]),
                       amax=g.float("amax", (len(counts),), torch.float32))
    if discrete:
        # each expert's codes and scales in an allocation of its own, allocated in reverse order
        per_sf = sfb.numel() // len(counts)
        # N-major: expert g's codes stored (k, n), the same values transposed
        b_list = [(qb[g].t().contiguous() if b_major == "n" else qb[g].clone())
                  for g in reversed(range(len(counts)))][::-1]
        sfb_list = [sfb[g * per_sf:(g + 1) * per_sf].clone() for g in reversed(range(len(counts)))][::-1]
        ws = torch.zeros(bsg.bsg_grouped_discrete_workspace_size(len(counts)), dtype=torch.uint8, device="cuda")
        out = torch_ops.grouped_gemm_srelu_discrete(
            qa[0], b_list, sfa, sfb_list, fmt, torch.from_numpy(offs).cuda(), torch.from_numpy(alpha).cuda(),
            torch.from_numpy(prob).cuda(), n, k, tanh_clamp_scale=clamp, d_dtype=d_dtype, c_dtype=c_dtype,
            norm_const=torch.tensor([nc], dtype=torch.float32, device="cuda"), workspace=ws, tile_n=tile_n,
            tanh_approx=tanh_approx, max_ctas=max_ctas, cta_pair=cta_pair, b_major=b_major, outputs=outputs)
    else:
        out = torch_ops.grouped_gemm_srelu(
            qa[0], qb, sfa, sfb, fmt, torch.from_numpy(offs).cuda(), torch.from_numpy(alpha).cuda(),
            torch.from_numpy(prob).cuda(), n, k, tanh_clamp_scale=clamp, d_dtype=d_dtype, c_dtype=c_dtype,
            norm_const=torch.tensor([nc], dtype=torch.float32, device="cuda"), workspace=ws, tile_n=tile_n,
            tanh_approx=tanh_approx, max_ctas=max_ctas, cta_pair=cta_pair, outputs=outputs)
    torch.cuda.synchronize()
    g.check()
    assert bsg.bsg_read_device_error(ws) == 0
    qa_ref, sfa_ref = oq.quantize(a, fmt)
    qb_ref, sfb_ref = oq.quantize(b, fmt)
    assert np.array_equal(qa.cpu().numpy(), qa_ref) and np.array_equal(qb.cpu().numpy(), qb_ref)
    assert np.array_equal(sfa.cpu().numpy(), sfa_ref) and np.array_equal(sfb.cpu().numpy(), sfb_ref)
    ref = og.grouped_srelu(qa_ref[0], qb_ref, sfa_ref, sfb_ref, fmt, offs, alpha, prob, k, n,
                           tanh_clamp_scale=clamp, d_fp8=(d_dtype == "e4m3"), norm_const=nc)
    # sum_k |Ahat||Bhat| per element for the tolerance, with each row's expert
    ahat = np.abs(oq.dequantize(qa_ref, sfa_ref, fmt, vm, k, 1)[0])
    bhat = np.abs(oq.dequantize(qb_ref, sfb_ref, fmt, n, k, len(counts)))
    g_of = og.expert_of_rows(offs, vm)
    s = np.zeros((vm, n))
    for g in range(len(counts)):
        rows = g_of == g
        if rows.any():
            s[rows] = float(alpha[g]) * (ahat[rows] @ bhat[g].T)
    c_tol = TOL_C * s
    if c_kind is not None:
        check_c_float(out["c"].float().cpu().numpy(), ref["c"], s, c_kind)
    d_tol = d_tolerance(ref["c"], prob, c_tol) + 2.0 ** -20 * ref["d"]
    if tanh_approx and clamp is not None:
        # the approximate tanh (max abs error 7.7e-6 on the pages' sweep) through d(c^2) = 2c dc
        d_tol = d_tol + np.asarray(prob, np.float64)[:, None] * 2 * clamp * clamp * 7.7e-6
    if d_dtype in ("bf16", "f16", "f32"):
        d_gpu = out["d"].float().cpu().numpy()
        if tanh_approx and clamp is not None:
            err = np.abs(d_gpu - ref["d"])
            assert np.all(err <= formats.bf16_ulp(ref["d"]) + d_tol)
        else:
            check_d_float(d_gpu, ref["d"], ref["c"], prob, c_tol, d_dtype)
        amax = out["amax"].cpu().numpy()
        assert np.all(amax[ref["amax"] == 0] == 0)
        nz = ref["amax"] > 0
        if tanh_approx and clamp is not None:
            assert np.allclose(amax[nz], ref["amax"][nz], rtol=2e-5)
        else:
            check_amax(amax[nz], ref["amax"][nz])
    else:
        sfd_row = sf_layout.unpack(out["sfd_row"].cpu().numpy(), vm, n // 32)[0]
        sfd_col = sf_layout.unpack(out["sfd_col"].cpu().numpy(), n, vm // 32)[0]
        nr = check_e4m3_blocks(out["d"].cpu().numpy(), sfd_row, ref["d"], d_tol, nc, axis=1, what="D_row")
        nc_ = check_e4m3_blocks(out["d_col"].cpu().numpy(), sfd_col, ref["d"], d_tol, nc, axis=0, what="D_col")
        # padding bytes of the SF buffers are zero
        full_row = out["sfd_row"].cpu().numpy()
        full_col = out["sfd_col"].cpu().numpy()
        assert (full_row != 0).sum() <= vm * (n // 32) and (full_col != 0).sum() <= n * (vm // 32)
        assert np.array_equal(sf_layout.pack(sfd_row[None]), full_row)
        assert np.array_equal(sf_layout.pack(sfd_col[None]), full_col)
        return out, ref, (nr, nc_)
    return out, ref, None


EDGE = [0, 300, 0, 0, 1, 256, 0]  # empty experts first, in a run and last; one 1-row expert


@pytest.mark.parametrize("counts,n,k,tile_n", [
    (EDGE, 256, 256, 0),
    (EDGE, 264, 512, 256),    # ragged N tile
    ([200, 200, 200, 200], 512, 384, 128),
    ([512], 384, 256, 256),   # single expert
    ([1, 2, 3, 700, 4], 256, 1024, 256),
    (EDGE, 704, 512, 224),    # tiles starting inside a 128-row scale atom
    ([200, 200, 200, 200], 600, 384, 192),
])
def test_grouped_bf16_d(lib, counts, n, k, tile_n):
    run_grouped(counts, n, k, "bf16", None, "bf16", tile_n=tile_n)


@pytest.mark.parametrize("counts,n,k,tile_n,cta_pair", [
    (EDGE, 256, 256, 0, 0),
    (EDGE, 264, 512, 256, 1),     # ragged N tile
    ([200, 200, 200, 200], 512, 384, 128, 1),
    ([1, 2, 3, 700, 4], 512, 1024, 0, 2),
])
def test_grouped_nvfp4_bf16_d(lib, counts, n, k, tile_n, cta_pair):
    run_grouped(counts, n, k, "bf16", None, "bf16", tile_n=tile_n, cta_pair=cta_pair, fmt="nvfp4")


def test_grouped_nvfp4_tanh_clamp(lib):
    run_grouped([300, 500, 0, 220], 256, 512, "bf16", 32.0, "f32", a_scale=700.0, fmt="nvfp4")


@pytest.mark.parametrize("fmt,d_dtype,c_kind,clamp,cta_pair", [
    ("mxfp8", "f16", "f16", None, 1),
    ("mxfp8", "f32", "f32", 32.0, 2),
    ("nvfp4", "f16", None, None, 2),
    ("nvfp4", "f32", "f16", 32.0, 1),
])
def test_grouped_d_types(lib, fmt, d_dtype, c_kind, clamp, cta_pair):
    run_grouped([300, 500, 0, 220], 256, 512, d_dtype, clamp, c_kind, cta_pair=cta_pair, fmt=fmt,
                a_scale=700.0 if clamp else 1.0)


def test_grouped_bf16_c_f32_and_no_c(lib):
    run_grouped(EDGE, 256, 256, "bf16", None, "f32")
    run_grouped(EDGE, 256, 256, "bf16", None, None)


@pytest.mark.parametrize("approx", [False, True])
def test_grouped_tanh_clamp(lib, approx):
    # inputs scaled so that |C| reaches well past s = 32 and the clamp saturates
    run_grouped([300, 500, 0, 220], 256, 512, "bf16", 32.0, "bf16", a_scale=700.0, tanh_approx=approx)


@pytest.mark.parametrize("nc,tile_n", [(1.0, 256), (1.0, 128), (0.75, 256), (1.0, 224), (0.75, 192)])
def test_grouped_fp8_d(lib, nc, tile_n):
    run_grouped(EDGE, 384, 512, "e4m3", None, "bf16", nc=nc, tile_n=tile_n)


def test_grouped_fp8_d_ragged_n_and_clamp(lib):
    run_grouped([257, 0, 511], 160, 256, "e4m3", 32.0, None, a_scale=700.0)


def test_grouped_few_ctas(lib):
    run_grouped([600, 900, 0, 300], 512, 512, "bf16", None, "bf16", tile_n=256, max_ctas=3)
    run_grouped([600, 900, 0, 300], 512, 512, "e4m3", None, "bf16", tile_n=128, max_ctas=2)


def test_grouped_bad_offsets_detected_on_device(lib):
    """Offsets that are not multiples of 256 are flagged on the device, nothing is computed."""
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg
    k, n, vm = 256, 256, 512
    qa = torch.zeros((vm, k), dtype=torch.uint8, device="cuda")
    qb = torch.zeros((2, n, k), dtype=torch.uint8, device="cuda")
    sfa = torch.zeros(bsg.bsg_sf_bytes(1, vm, k, 32), dtype=torch.uint8, device="cuda")
    sfb = torch.zeros(bsg.bsg_sf_bytes(2, n, k, 32), dtype=torch.uint8, device="cuda")
    ws = torch_ops.new_workspace()
    offs = torch.tensor([100, 512], dtype=torch.int32, device="cuda")
    ones = torch.ones(2, device="cuda")
    prob = torch.ones(vm, device="cuda")
    torch_ops.grouped_gemm_srelu(qa, qb, sfa, sfb, "mxfp8", offs, ones, prob, n, k, workspace=ws)
    assert bsg.bsg_read_device_error(ws) == bsg.DEVERR_BAD_OFFSETS
    with pytest.raises(bsg.BsgError) as ei:
        torch_ops.grouped_gemm_srelu(qa, qb, sfa, sfb, "mxfp8", offs, ones, prob, n, k, workspace=ws,
                                     validate_offsets=True)
    assert ei.value.status == 7


@pytest.mark.parametrize("d_dtype,clamp,c_kind,n,nc", [
    ("bf16", None, "bf16", 256, 1.0),
    ("bf16", 32.0, "f32", 264, 1.0),    # ragged N
    ("e4m3", None, "bf16", 384, 1.0),
    ("e4m3", None, None, 512, 0.75),
    # bf16 D (with bf16 or no C) on pairs: blocks stored by TMA, clipped at ragged N
    ("bf16", None, None, 264, 1.0),
    ("bf16", 32.0, "bf16", 520, 1.0),
])
def test_grouped_cta_pairs(lib, d_dtype, clamp, c_kind, n, nc):
    run_grouped(EDGE, n, 512, d_dtype, clamp, c_kind, nc=nc, cta_pair=2, a_scale=700.0 if clamp else 1.0)


@pytest.mark.parametrize("d_dtype,clamp,n", [("e4m3", None, 384), ("e4m3", 32.0, 704), ("bf16", None, 704)])
def test_grouped_cta_pairs_224(lib, d_dtype, clamp, n):
    run_grouped(EDGE, n, 512, d_dtype, clamp, "bf16", tile_n=224, cta_pair=2, a_scale=700.0 if clamp else 1.0)


def test_grouped_cta_pairs_few_clusters(lib):
    run_grouped([600, 900, 0, 300], 512, 512, "bf16", None, "bf16", cta_pair=2, max_ctas=2)
    run_grouped([600, 900, 0, 300], 512, 512, "e4m3", None, "bf16", cta_pair=2, max_ctas=4)


@pytest.mark.parametrize("fmt,d_dtype,clamp,n,tile_n,cta_pair", [
    ("mxfp8", "bf16", None, 264, 256, 1),    # ragged N, one-CTA tiles
    ("mxfp8", "bf16", 32.0, 512, 0, 2),      # CTA pairs
    ("mxfp8", "e4m3", None, 384, 224, 2),    # FP8 D on 224-wide pair tiles
    ("mxfp8", "e4m3", None, 384, 128, 1),
    ("nvfp4", "bf16", None, 512, 0, 2),
    ("nvfp4", "f16", None, 264, 128, 1),
])
def test_grouped_discrete_weights(lib, fmt, d_dtype, clamp, n, tile_n, cta_pair):
    """Per-expert weight allocations addressed by pointer arrays give the contiguous form's result."""
    run_grouped(EDGE, n, 512, d_dtype, clamp, "bf16", tile_n=tile_n, cta_pair=cta_pair, fmt=fmt,
                a_scale=700.0 if clamp else 1.0, discrete=True)


@pytest.mark.parametrize("counts,d_dtype,clamp,n,k,tile_n,cta_pair", [
    (EDGE, "bf16", None, 512, 512, 0, 2),        # 256-wide CTA pairs (128 N per CTA)
    (EDGE, "e4m3", None, 384, 512, 0, 2),        # E4M3 D on N-major B: pairs, ragged last N tile
    (EDGE, "bf16", 32.0, 272, 320, 128, 1),      # one-CTA 128-wide tiles, ragged N, K tail
    (EDGE, "e4m3", None, 256, 1024, 128, 1),
    ([600, 900, 0, 300], "bf16", None, 768, 256, 0, 2),
])
def test_grouped_discrete_weights_n_major(lib, counts, d_dtype, clamp, n, k, tile_n, cta_pair):
    """FP8 per-expert weights stored N-major, (k, n) with n contiguous ("Grouped GEMM + sReLU
    (SM100)", Support surface and constraints), give the oracle's result."""
    run_grouped(counts, n, k, d_dtype, clamp, "bf16", tile_n=tile_n, cta_pair=cta_pair, fmt="mxfp8",
                a_scale=700.0 if clamp else 1.0, discrete=True, b_major="n")


def test_grouped_discrete_n_major_rejections(lib):
    """N-major B: MXFP8 only, per-expert weights only, 128 / 256-wide tiles, n % 16 == 0."""
    import nvfp4_gemm_moe_gb300 as bsg
    from nvfp4_gemm_moe_gb300 import torch_ops
    k, n, vm = 256, 256, 256
    qa = torch.zeros((vm, k), dtype=torch.uint8, device="cuda")
    sfa = torch.zeros(bsg.bsg_sf_bytes(1, vm, k, 32), dtype=torch.uint8, device="cuda")
    bs = [torch.zeros((k, n), dtype=torch.uint8, device="cuda")]
    sfbs = [torch.zeros(bsg.bsg_sf_bytes(1, n, k, 32), dtype=torch.uint8, device="cuda")]
    offs = torch.tensor([vm], dtype=torch.int32, device="cuda")
    one, prob = torch.ones(1, device="cuda"), torch.ones(vm, device="cuda")
    with pytest.raises(bsg.BsgError) as ei:
        torch_ops.grouped_gemm_srelu_discrete(qa, bs, sfa, sfbs, "mxfp8", offs, one, prob, n, k, b_major="n",
                                              tile_n=224, cta_pair=2)
    assert ei.value.status == 2
    with pytest.raises(bsg.BsgError) as ei:
        torch_ops.grouped_gemm_srelu(qa, bs[0][None], sfa, sfbs[0], "mxfp8", offs, one, prob, n, k, b_major="n")
    assert ei.value.status == 1
    with pytest.raises(bsg.BsgError) as ei:
        torch_ops.grouped_gemm_srelu_discrete(qa, [torch.zeros((k, n // 2), dtype=torch.uint8, device="cuda")], sfa,
                                              [torch.zeros(bsg.bsg_sf_bytes(1, n, k, 16), dtype=torch.uint8,
                                                           device="cuda")], "nvfp4", offs, one, prob, n, k,
                                              b_major="n")
    assert ei.value.status == 2


def test_grouped_discrete_pointer_validation(lib):
    """Null or misaligned pointer entries are found on the device: the call records
    BSG_DEVERR_BAD_POINTERS and writes nothing (D stays poisoned, amax zero); a short workspace is
    rejected on the host; the next call with good pointers on the same workspace runs clean."""
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg
    k, n, vm = 256, 256, 512
    qa = torch.zeros((vm, k), dtype=torch.uint8, device="cuda")
    bs = [torch.zeros((n, k), dtype=torch.uint8, device="cuda") for _ in range(2)]
    sfa = torch.zeros(bsg.bsg_sf_bytes(1, vm, k, 32), dtype=torch.uint8, device="cuda")
    sfbs = [torch.zeros(bsg.bsg_sf_bytes(1, n, k, 32), dtype=torch.uint8, device="cuda") for _ in range(2)]
    offs = torch.tensor([256, 512], dtype=torch.int32, device="cuda")
    ones = torch.ones(2, device="cuda")
    prob = torch.ones(vm, device="cuda")
    good_b = torch.tensor([t.data_ptr() for t in bs], dtype=torch.int64, device="cuda")
    good_s = torch.tensor([t.data_ptr() for t in sfbs], dtype=torch.int64, device="cuda")
    bad_cases = [
        (torch.tensor([bs[0].data_ptr(), 0], dtype=torch.int64, device="cuda"), good_s),
        (good_b, torch.tensor([0, sfbs[1].data_ptr()], dtype=torch.int64, device="cuda")),
        (torch.tensor([bs[0].data_ptr() + 8, bs[1].data_ptr()], dtype=torch.int64, device="cuda"), good_s),
        (good_b, torch.tensor([sfbs[0].data_ptr(), sfbs[1].data_ptr() + 4], dtype=torch.int64, device="cuda")),
    ]
    ws = torch.zeros(bsg.bsg_grouped_discrete_workspace_size(2), dtype=torch.uint8, device="cuda")
    for bp, sp in bad_cases:
        out = {"d": torch.full((vm, n), float("nan"), dtype=torch.bfloat16, device="cuda"),
               "amax": torch.full((2,), -1.0, device="cuda"), "c": None}
        bsg.bsg_grouped_gemm_srelu_discrete(qa, bp, sfa, sp, bsg.E4M3, bsg.SF_UE8M0, 32, vm, n, k, 2, offs, ones,
                                            prob, None, None, None, bsg.BF16, out["d"], None, bsg.BF16, None,
                                            None, out["amax"], ws)
        assert bsg.bsg_read_device_error(ws) == bsg.DEVERR_BAD_POINTERS
        assert torch.isnan(out["d"].float()).all() and torch.equal(out["amax"].cpu(), torch.zeros(2))
    with pytest.raises(bsg.BsgError) as ei:
        bsg.bsg_grouped_gemm_srelu_discrete(qa, good_b, sfa, good_s, bsg.E4M3, bsg.SF_UE8M0, 32, vm, n, k, 2, offs,
                                            ones, prob, None, None, None, bsg.BF16, out["d"], None, bsg.BF16, None,
                                            None, out["amax"], ws, workspace_bytes=bsg.bsg_workspace_size())
    assert ei.value.status == 8
    # the good pointers run on the same workspace and give zeros, with no device error
    out = torch_ops.grouped_gemm_srelu_discrete(qa, good_b, sfa, good_s, "mxfp8", offs, ones, prob, n, k, workspace=ws)
    torch.cuda.synchronize()
    assert bsg.bsg_read_device_error(ws) == 0
    assert float(out["d"].float().abs().max()) == 0.0


def test_grouped_max_experts(lib):
    """1024 experts (the limit the kernel stages in shared memory), all but three empty."""
    counts = [0] * 1024
    counts[0], counts[517], counts[1023] = 40, 300, 256
    run_grouped(counts, 256, 256, "bf16", None, "bf16")


def test_grouped_all_experts_empty(lib):
    """valid_m = 0: nothing to compute, the per-expert amax is zeroed, no kernel error."""
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg
    k, n, num_experts = 256, 256, 4
    qa = torch.zeros((0, k), dtype=torch.uint8, device="cuda")  # empty: its data pointer may be null
    qb = torch.zeros((num_experts, n, k), dtype=torch.uint8, device="cuda")
    sfa = torch.zeros(512, dtype=torch.uint8, device="cuda")
    sfb = torch.zeros(bsg.bsg_sf_bytes(num_experts, n, k, 32), dtype=torch.uint8, device="cuda")
    offs = torch.zeros(num_experts, dtype=torch.int32, device="cuda")
    ws = torch_ops.new_workspace()
    amax = torch.full((num_experts,), float("nan"), device="cuda")
    out = torch_ops.grouped_gemm_srelu(qa, qb, sfa, sfb, "mxfp8", offs, torch.ones(num_experts, device="cuda"),
                                       torch.ones(1, device="cuda"), n, k, workspace=ws,
                                       outputs={"amax": amax, "c": None,
                                                "d": torch.zeros((0, n), dtype=torch.bfloat16, device="cuda")})
    torch.cuda.synchronize()
    assert bsg.bsg_read_device_error(ws) == 0
    assert torch.all(out["amax"] == 0)

"""GPU parity of bsg_gemm_amax (dense / batched block-scaled GEMM + global amax) against the oracle.

Both paths start from the same seeded fp32 operands; each quantises them with its own
quantiser (asserted bit-identical first), then the GPU GEMM is compared element by
element with the float64 oracle on shapes that span several tiles and ragged tails.
"""
import numpy as np
import pytest
import torch

from guards import Outputs

import workloads as W
from oracle import gemm as og, quantize as oq
from parity import TOL_C, check_amax, check_c_float, check_codes_plain

pytestmark = pytest.mark.gpu


def _operands(seed, fmt, m, n, k, l, boost=False, spread=False):
    a = W.normal_f32(seed, W.S_A, 0, l * m * k).reshape(l, m, k)
    b = W.normal_f32(seed, W.S_B, 0, l * n * k).reshape(l, n, k)
    if boost:
        v = 32 if fmt == "mxfp8" else 16
        kb = np.arange(k) // v
        a[..., kb % 7 == 6] *= np.float32(64.0)
    if spread:
        e = np.clip(np.round(W.normal_f32(seed, 21, 0, l * m) * 6), -30, 30).reshape(l, m, 1)
        a = (a * np.exp2(e)).astype(np.float32)
    return a, b


def run_dense(fmt, m, n, k, l, c_kind, tile_n=0, seed=1, boost=False, spread=False, max_ctas=0, cta_pair=0):
    from nvfp4_gemm_moe_gb300 import torch_ops
    a, b = _operands(seed, fmt, m, n, k, l, boost, spread)
    qa, sfa = torch_ops.quantize(torch.from_numpy(a).cuda(), fmt)
    qb, sfb = torch_ops.quantize(torch.from_numpy(b).cuda(), fmt)
    c_dtype = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16, "e4m3": "e4m3", "e2m1": "e2m1"}[c_kind]
    ws = torch_ops.new_workspace()
    g = Outputs()
    if c_kind in ("e4m3", "e2m1"):
        c_out = g.codes("c", (l, m, n if c_kind == "e4m3" else n // 2))
    else:
        c_out = g.float("c", (l, m, n), c_dtype)
    amax_out = g.float("amax", (1,), torch.float32)
    c, amax = torch_ops.gemm_amax(qa, qb, sfa, sfb, fmt, m, n, k, l, c_dtype=c_dtype, c=c_out, amax=amax_out,
                                  workspace=ws, tile_n=tile_n, max_ctas=max_ctas, cta_pair=cta_pair)
    torch.cuda.synchronize()
    g.check()
    import nvfp4_gemm_moe_gb300 as bsg
    assert bsg.bsg_read_device_error(ws) == 0
    # oracle side
    qa_ref, sfa_ref = oq.quantize(a, fmt)
    qb_ref, sfb_ref = oq.quantize(b, fmt)
    assert np.array_equal(qa.cpu().numpy().reshape(qa_ref.shape), qa_ref)
    assert np.array_equal(qb.cpu().numpy().reshape(qb_ref.shape), qb_ref)
    assert np.array_equal(sfa.cpu().numpy(), sfa_ref) and np.array_equal(sfb.cpu().numpy(), sfb_ref)
    ref, amax_ref = og.dense_gemm_amax(qa_ref, qb_ref, sfa_ref, sfb_ref, fmt, m, n, k, l)
    s = og.dense_abs_sum(qa_ref, qb_ref, sfa_ref, sfb_ref, fmt, m, n, k, l)
    if c_kind in ("e4m3", "e2m1"):
        check_codes_plain(c.cpu().numpy(), ref, TOL_C * s, c_kind)
    else:
        check_c_float(c.float().cpu().numpy(), ref, s, c_kind)
    check_amax(amax.cpu().numpy()[0], amax_ref)
    return c, amax


@pytest.mark.parametrize("fmt,m,n,k,l,c_kind,tile_n", [
    ("mxfp8", 256, 256, 256, 1, "f32", 0),      # the small dense workload's shape
    ("mxfp8", 256, 256, 256, 1, "f32", 256),
    ("mxfp8", 300, 264, 384, 2, "bf16", 0),     # ragged M and N, batch 2
    ("mxfp8", 384, 520, 1024, 1, "bf16", 256),  # several N tiles, ragged last one
    ("mxfp8", 384, 520, 1024, 1, "f32", 128),
    ("mxfp8", 128, 128, 160, 1, "f32", 128),    # K tail: one 32-wide MMA in the last stage
    ("mxfp8", 1, 8, 32, 1, "f32", 128),         # minimal
    ("mxfp8", 384, 1000, 512, 1, "bf16", 224),  # tiles starting inside a 128-row scale atom
    ("mxfp8", 256, 640, 256, 2, "f32", 192),
    ("nvfp4", 256, 256, 512, 1, "bf16", 256),
    ("nvfp4", 300, 264, 320, 2, "f32", 128),    # K tail: one MMA in the last stage
    ("nvfp4", 130, 136, 96, 1, "f32", 0),       # K = 96: half of the second MMA is zero fill
    ("nvfp4", 640, 768, 2048, 1, "bf16", 256),
])
def test_dense_parity(lib, fmt, m, n, k, l, c_kind, tile_n):
    run_dense(fmt, m, n, k, l, c_kind, tile_n)


def test_dense_scale_range_boosted_blocks(lib):
    """Every 7th K block of A x2^6 and rows spread over 2^+-30 (E8M0 scale range)."""
    run_dense("mxfp8", 512, 384, 2048, 2, "bf16", 256, boost=True, spread=True)
    run_dense("nvfp4", 256, 384, 1024, 1, "f32", 128, boost=True)


def test_dense_persistent_loop_few_ctas(lib):
    """Few CTAs: each walks many tiles, exercising stage / accumulator phase wrap-around."""
    run_dense("mxfp8", 1024, 1024, 1024, 1, "bf16", 256, max_ctas=3)
    run_dense("mxfp8", 1024, 1024, 512, 1, "f32", 128, max_ctas=5)
    run_dense("nvfp4", 512, 768, 1024, 1, "bf16", 256, max_ctas=2)


def test_dense_repeat_calls_are_identical(lib):
    c1, a1 = run_dense("mxfp8", 256, 512, 512, 1, "bf16", 256, seed=7)
    c2, a2 = run_dense("mxfp8", 256, 512, 512, 1, "bf16", 256, seed=7)
    assert torch.equal(c1, c2) and torch.equal(a1, a2)


@pytest.mark.parametrize("fmt,m,n,k,l,c_kind", [
    ("mxfp8", 256, 256, 256, 1, "f32"),
    ("mxfp8", 300, 264, 384, 2, "bf16"),     # ragged M (second 256-row tile mostly empty) and N
    ("mxfp8", 512, 768, 1024, 1, "bf16"),
    ("mxfp8", 256, 256, 160, 1, "f32"),      # K tail
    ("nvfp4", 256, 256, 512, 1, "bf16"),
    ("nvfp4", 300, 264, 320, 2, "f32"),      # K tail: one MMA in the last stage
    ("nvfp4", 512, 512, 2048, 1, "bf16"),
])
def test_dense_parity_cta_pairs(lib, fmt, m, n, k, l, c_kind):
    run_dense(fmt, m, n, k, l, c_kind, cta_pair=2)


@pytest.mark.parametrize("m,n,k,l,c_kind", [
    (512, 1000, 512, 1, "bf16"),   # 224-wide pair tiles starting inside a 128-row scale atom
    (300, 448, 384, 2, "f32"),
])
def test_dense_parity_cta_pairs_224(lib, m, n, k, l, c_kind):
    run_dense("mxfp8", m, n, k, l, c_kind, tile_n=224, cta_pair=2)


@pytest.mark.parametrize("fmt,m,n,k,l,c_kind,cta_pair", [
    ("mxfp8", 300, 264, 384, 2, "f16", 1),
    ("mxfp8", 512, 512, 512, 1, "f16", 2),
    ("nvfp4", 300, 264, 320, 2, "f16", 1),
    ("nvfp4", 256, 256, 512, 1, "e4m3", 1),   # plain FP8 C with FP4 operands
    ("nvfp4", 512, 512, 512, 1, "e4m3", 2),
    ("nvfp4", 256, 320, 512, 1, "e2m1", 1),   # packed FP4 C
    ("nvfp4", 512, 512, 1024, 2, "e2m1", 2),
])
def test_dense_c_types(lib, fmt, m, n, k, l, c_kind, cta_pair):
    run_dense(fmt, m, n, k, l, c_kind, cta_pair=cta_pair)


def test_dense_c_type_rejections(lib):
    import nvfp4_gemm_moe_gb300 as bsg
    from nvfp4_gemm_moe_gb300 import torch_ops
    q = torch.zeros((1, 256, 256), dtype=torch.uint8, device="cuda")
    sf = torch.zeros(bsg.bsg_sf_bytes(1, 256, 256, 32), dtype=torch.uint8, device="cuda")
    for ck in ("e4m3", "e2m1"):  # FP8 C with FP8 operands is disabled; FP4 C needs FP4 operands
        with pytest.raises(bsg.BsgError) as ei:
            torch_ops.gemm_amax(q, q, sf, sf, "mxfp8", 256, 256, 256, 1, c_dtype=ck)
        assert ei.value.status == 2  # BSG_ERR_UNSUPPORTED


def test_dense_cta_pairs_few_clusters(lib):
    """Two pairs walk many 256 x 256 tiles: stage and accumulator phases wrap around."""
    run_dense("mxfp8", 1024, 1024, 1024, 2, "bf16", cta_pair=2, max_ctas=4, boost=True)
    run_dense("nvfp4", 768, 1024, 1024, 1, "bf16", cta_pair=2, max_ctas=2)


@pytest.mark.parametrize("cta_pair,max_ctas", [(1, 0), (1, 1), (2, 0), (2, 2)])
def test_dense_amax_from_stale_workspace(lib, cta_pair, max_ctas):
    """The kernel writes amax itself (the last CTA to finish) from a reduction it keeps in the
    workspace under the call's tag: a workspace full of another call's leftovers (bytes 0xA5) and
    a poisoned amax give the oracle's amax and no device error, twice in a row, on one CTA, one
    pair, and full grids of CTAs and pairs."""
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg
    fmt, m, n, k, l = "mxfp8", 640, 512, 256, 2
    a, b = _operands(5, fmt, m, n, k, l, spread=True)
    qa, sfa = torch_ops.quantize(torch.from_numpy(a).cuda(), fmt)
    qb, sfb = torch_ops.quantize(torch.from_numpy(b).cuda(), fmt)
    qa_ref, sfa_ref = oq.quantize(a, fmt)
    qb_ref, sfb_ref = oq.quantize(b, fmt)
    _, amax_ref = og.dense_gemm_amax(qa_ref, qb_ref, sfa_ref, sfb_ref, fmt, m, n, k, l)
    ws = torch.full((bsg.bsg_workspace_size(),), 0xA5, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        amax = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
        torch_ops.gemm_amax(qa, qb, sfa, sfb, fmt, m, n, k, l, c_dtype=torch.float32, amax=amax, workspace=ws,
                            cta_pair=cta_pair, max_ctas=max_ctas)
        torch.cuda.synchronize()
        check_amax(amax.cpu().numpy(), np.array([amax_ref]))
        assert bsg.bsg_read_device_error(ws) == 0

"""bsg_gemm_amax_noalloc: the dense GEMM + amax for callers that cannot provide device memory.

Callers running under a start-up memory plan that forbids later allocations, or on a
latency-critical path that cannot afford cudaMalloc's implicit synchronisation, cannot hand
the library a workspace.  This entry point keeps its scratch in a static device array of the
library instead.  The test calls it through the C ABI twice in a row on the same inputs and
checks both results against the float64 oracle with the dense parity tests' tolerance
(|C - ref| <= 2^-20 sum_k |Ahat||Bhat|, amax within 1e-5 relative), and that each call left
no device error in the library's array.  The file sorts last so that a run stopping at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import gemm as og, quantize as oq

pytestmark = pytest.mark.gpu


def test_noalloc_matches_oracle_twice(lib):
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg

    for fmt, m, n, k, l in (("mxfp8", 300, 264, 512, 2), ("nvfp4", 256, 384, 1024, 1)):
        a = W.normal_f32(31, W.S_A, 0, l * m * k).reshape(l, m, k)
        b = W.normal_f32(31, W.S_B, 0, l * n * k).reshape(l, n, k)
        qa, sfa = torch_ops.quantize(torch.from_numpy(a).cuda(), fmt)
        qb, sfb = torch_ops.quantize(torch.from_numpy(b).cuda(), fmt)
        ab, sfd, v = bsg.FORMATS[fmt]
        qa_o, sfa_o = oq.quantize(a, fmt)
        qb_o, sfb_o = oq.quantize(b, fmt)
        ref, amax_ref = og.dense_gemm_amax(qa_o, qb_o, sfa_o, sfb_o, fmt, m, n, k, l)
        bound = 2.0 ** -20 * og.dense_abs_sum(qa_o, qb_o, sfa_o, sfb_o, fmt, m, n, k, l)
        for _ in range(2):
            c = torch.full((l, m, n), float("nan"), dtype=torch.float32, device="cuda")
            amax = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
            bsg.bsg_gemm_amax_noalloc(qa, qb, sfa, sfb, ab, sfd, v, m, n, k, l, c, bsg.F32, amax)
            assert bsg.bsg_gemm_amax_noalloc_read_error() == 0
            err = np.abs(c.cpu().numpy().astype(np.float64) - ref)
            assert np.all(err <= bound)
            assert abs(float(amax.item()) - amax_ref) <= 1e-5 * amax_ref

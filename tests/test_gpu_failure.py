"""Device-side failure detection without a GPU fault: a bounded wait that runs out.

The self-test kernel waits on an mbarrier that nothing arrives on, with the same bounded wait
the GEMM roles use; after the 2 s limit it records BSG_DEVERR_TIMEOUT and returns.  The test
reads the error bits on the host and then runs a GEMM on the same context and workspace to show
that the context is still usable and that the GEMM's error record replaces the timed-out one.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import gemm as og, quantize as oq

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_stays_usable(lib):
    from nvfp4_gemm_moe_gb300 import torch_ops
    import nvfp4_gemm_moe_gb300 as bsg
    ws = torch_ops.new_workspace()
    bsg.bsg_selftest_wait_timeout(ws)
    assert bsg.bsg_read_device_error(ws) == bsg.DEVERR_TIMEOUT
    # the context still runs kernels: the small dense GEMM against the oracle
    wl = W.DENSE_MXFP8_256
    a, b = wl.a_rows(), wl.b_rows()
    qa, sfa = torch_ops.quantize(torch.from_numpy(a).cuda(), "mxfp8")
    qb, sfb = torch_ops.quantize(torch.from_numpy(b).cuda(), "mxfp8")
    c, amax = torch_ops.gemm_amax(qa, qb, sfa, sfb, "mxfp8", wl.m, wl.n, wl.k, wl.l, c_dtype=torch.float32,
                                  workspace=ws)
    torch.cuda.synchronize()
    assert bsg.bsg_read_device_error(ws) == 0
    qa_r, sfa_r = oq.quantize(a, "mxfp8")
    qb_r, sfb_r = oq.quantize(b, "mxfp8")
    ref, amax_ref = og.dense_gemm_amax(qa_r, qb_r, sfa_r, sfb_r, "mxfp8", wl.m, wl.n, wl.k, wl.l)
    s = og.dense_abs_sum(qa_r, qb_r, sfa_r, sfb_r, "mxfp8", wl.m, wl.n, wl.k, wl.l)
    assert np.all(np.abs(c.cpu().numpy().astype(np.float64) - ref) <= 2.0 ** -20 * s)
    # the timed-out call's bits stay behind in the workspace, tagged with its number: the GEMM's
    # own (empty) record replaced them, and its amax reduction there ignored them
    assert abs(float(amax.item()) - amax_ref) <= 1e-5 * amax_ref

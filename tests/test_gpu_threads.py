"""The library from two host threads at once: each thread drives its own stream and workspace
through the NVFP4 quantiser and a one-CTA dense GEMM (in a fresh process, the first launches
of both kernels race); every result must equal the same calls made from one thread."""
import threading

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def _work(seed, stream, results, key):
    from nvfp4_gemm_moe_gb300 import torch_ops
    with torch.cuda.stream(stream):
        a = torch.from_numpy(W.normal_f32(seed, W.S_A, 0, 384 * 640).reshape(1, 384, 640)).cuda()
        b = torch.from_numpy(W.normal_f32(seed, W.S_B, 0, 512 * 640).reshape(1, 512, 640)).cuda()
        ws = torch_ops.new_workspace()
        outs = []
        for _ in range(10):
            qa, sfa = torch_ops.quantize(a, "nvfp4")
            qb, sfb = torch_ops.quantize(b, "nvfp4")
            c, amax = torch_ops.gemm_amax(qa, qb, sfa, sfb, "nvfp4", 384, 512, 640, 1, c_dtype=torch.float32,
                                          workspace=ws, tile_n=128, cta_pair=1)
            outs.append((c, amax))
        stream.synchronize()
        results[key] = [(c.cpu(), amax.cpu()) for c, amax in outs]


def test_two_host_threads(lib):
    results = {}
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    threads = [threading.Thread(target=_work, args=(seed, streams[i], results, i)) for i, seed in enumerate((3, 4))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert sorted(results) == [0, 1]
    solo = {}
    _work(3, torch.cuda.Stream(), solo, 0)
    _work(4, torch.cuda.Stream(), solo, 1)
    for i in (0, 1):
        for (c, amax), (c_ref, amax_ref) in zip(results[i], solo[i]):
            assert torch.equal(c, c_ref) and torch.equal(amax, amax_ref)
    assert not np.isnan(results[0][0][0].numpy()).any()

"""The entry points under CUDA graph capture: quantise + dense GEMM, a grouped sReLU GEMM with
E4M3 D and a RoPE projection captured once on one stream, replayed on new input data; every
output must equal an eager call's on the same data, bit for bit (the kernels are deterministic:
fixed reduction orders, maxima folded with order-independent atomics)."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def _draw(seed, shape, scale=1.0):
    n = int(np.prod(shape))
    return torch.from_numpy(W.normal_f32(seed, W.S_A, 0, n).reshape(shape) * np.float32(scale))


def test_capture_and_replay_matches_eager(lib):
    from nvfp4_gemm_moe_gb300 import torch_ops
    dev = "cuda"
    m, n, k = 256, 384, 512
    g = W.Grouped("graph", 3, 256, 256, 700, "fixed:300,0,400", "bf16", seed=4)
    offs = torch.from_numpy(g.padded_offsets()).to(dev)
    alpha = torch.from_numpy(g.alpha()).to(dev)
    prob = torch.from_numpy(g.prob()).to(dev)
    nc = torch.ones(1, device=dev)
    tokens, q_lora, heads = 256, 256, 2
    cos32, sin32 = W.RopeProj("graph", tokens, q_lora, heads, 192, 64).tables()
    cos = torch.from_numpy(cos32).to(torch.bfloat16).to(dev)
    sin = torch.from_numpy(sin32).to(torch.bfloat16).to(dev)

    # static input buffers the graph reads at replay time
    a = torch.empty((1, m, k), device=dev)
    b = torch.empty((1, n, k), device=dev)
    ga = torch.empty((1, g.valid_m, g.k), device=dev)
    gb = torch.empty((g.experts, g.n, g.k), device=dev)
    x = torch.empty((tokens, q_lora), dtype=torch.bfloat16, device=dev)
    w = torch.empty((heads * 192, q_lora), dtype=torch.bfloat16, device=dev)
    ws = [torch_ops.new_workspace(dev) for _ in range(3)]

    def fill(seed):
        a.copy_(_draw(seed, (1, m, k)))
        b.copy_(_draw(seed + 1, (1, n, k)))
        ga.copy_(_draw(seed + 2, (1, g.valid_m, g.k)))
        gb.copy_(_draw(seed + 3, (g.experts, g.n, g.k), 1 / 16))
        x.copy_(_draw(seed + 4, (tokens, q_lora)).to(torch.bfloat16))
        w.copy_(_draw(seed + 5, (heads * 192, q_lora), 1 / 16).to(torch.bfloat16))

    outs = {}

    def step():
        qa, sfa = torch_ops.quantize(a, "mxfp8", q=outs.get("qa"), sf=outs.get("sfa"))
        qb, sfb = torch_ops.quantize(b, "mxfp8", q=outs.get("qb"), sf=outs.get("sfb"))
        outs.update(qa=qa, sfa=sfa, qb=qb, sfb=sfb)
        c, amax = torch_ops.gemm_amax(qa, qb, sfa, sfb, "mxfp8", m, n, k, 1, c=outs.get("c"), amax=outs.get("amax"),
                                      c_dtype=torch.bfloat16, workspace=ws[0])
        outs.update(c=c, amax=amax)
        gqa, gsfa = torch_ops.quantize(ga, "mxfp8", q=outs.get("gqa"), sf=outs.get("gsfa"))
        gqb, gsfb = torch_ops.quantize(gb, "mxfp8", q=outs.get("gqb"), sf=outs.get("gsfb"))
        outs.update(gqa=gqa, gsfa=gsfa, gqb=gqb, gsfb=gsfb)
        gout = torch_ops.grouped_gemm_srelu(gqa[0], gqb, gsfa, gsfb, "mxfp8", offs, alpha, prob, g.n, g.k,
                                            d_dtype="e4m3", norm_const=nc, outputs=outs.get("grouped"),
                                            workspace=ws[1])
        outs["grouped"] = gout
        outs["rope"] = torch_ops.gemm_rope_bf16(x, w, cos, sin, heads, outputs=outs.get("rope"), workspace=ws[2])

    def snapshot():
        keys = ("qa", "sfa", "qb", "sfb", "c", "amax")
        snap = {k2: outs[k2].clone() for k2 in keys}
        snap.update({"g_" + k2: v.clone() for k2, v in outs["grouped"].items()})
        snap.update({"r_" + k2: v.clone() for k2, v in outs["rope"].items()})
        return snap

    # eager results for two data sets (the first calls also set every kernel's attributes)
    fill(10)
    step()
    torch.cuda.synchronize()
    eager1 = snapshot()
    fill(20)
    step()
    torch.cuda.synchronize()
    eager2 = snapshot()

    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            step()
    torch.cuda.synchronize()

    for seed, ref in ((10, eager1), (20, eager2), (10, eager1)):
        fill(seed)
        graph.replay()
        torch.cuda.synchronize()
        got = snapshot()
        for key, v in ref.items():
            assert torch.equal(got[key], v), f"{key} differs after replay (data set {seed})"
    import nvfp4_gemm_moe_gb300 as bsg
    assert all(bsg.bsg_read_device_error(wk) == 0 for wk in ws)


def test_capture_discrete_weights(lib):
    """The per-expert-weight call captured in a graph: its TMA descriptors are rebuilt on the
    device from the pointer arrays at every replay, so new contents of the arrays (the experts'
    weights in another order) take effect on replay, equal to an eager call bit for bit."""
    from nvfp4_gemm_moe_gb300 import torch_ops
    dev = "cuda"
    g = W.Grouped("graph_discrete", 3, 256, 256, 700, "fixed:300,0,400", "bf16", seed=6)
    offs = torch.from_numpy(g.padded_offsets()).to(dev)
    alpha = torch.from_numpy(g.alpha()).to(dev)
    prob = torch.from_numpy(g.prob()).to(dev)
    qa, sfa = torch_ops.quantize(_draw(30, (1, g.valid_m, g.k)).to(dev), "mxfp8")
    experts = [torch_ops.quantize(_draw(31 + e, (1, g.n, g.k), 1 / 16).to(dev), "mxfp8") for e in range(g.experts)]
    ws = torch.zeros(lib.bsg_grouped_discrete_workspace_size(g.experts), dtype=torch.uint8, device=dev)
    bp = torch.empty(g.experts, dtype=torch.int64, device=dev)
    sp = torch.empty(g.experts, dtype=torch.int64, device=dev)

    def point(order):
        bp.copy_(torch.tensor([experts[e][0].data_ptr() for e in order], dtype=torch.int64))
        sp.copy_(torch.tensor([experts[e][1].data_ptr() for e in order], dtype=torch.int64))

    outs = {}

    def step():
        outs["o"] = torch_ops.grouped_gemm_srelu_discrete(qa[0], bp, sfa, sp, "mxfp8", offs, alpha, prob, g.n, g.k,
                                                          outputs=outs.get("o"), workspace=ws)

    eager = {}
    for order in ((0, 1, 2), (2, 0, 1)):
        point(order)
        step()
        torch.cuda.synchronize()
        eager[order] = {k2: v.clone() for k2, v in outs["o"].items() if v is not None}
    assert not torch.equal(eager[(0, 1, 2)]["d"], eager[(2, 0, 1)]["d"])
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            step()
    torch.cuda.synchronize()
    for order in ((2, 0, 1), (0, 1, 2), (2, 0, 1)):
        point(order)
        graph.replay()
        torch.cuda.synchronize()
        for key, v in eager[order].items():
            assert torch.equal(outs["o"][key], v), f"{key} differs after replay (order {order})"
    assert lib.bsg_read_device_error(ws) == 0

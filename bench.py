"""Throughput benchmark of the block-scaled GEMM hot path on GB300.

One step = the whole hot path over one batch of synthetic input: quantise A and B
(fp32 -> MXFP8 / NVFP4 codes + scale factors) and run the block-scaled GEMM with its
fused epilogue (bf16-operand workloads skip the quantisation: their step is the kernel
alone).  Default workload: the batched dense MXFP8 GEMM + amax, L = 4,
M = N = K = 8192, C bf16.  Inputs (2 x 1.07 GB fp32) are larger than L2, so no flush
is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs an independent replica
of the workload on its own GPU ("replicas only": the path has no exchange step); the
elapsed time is the maximum over ranks and `value` counts the work of all ranks.
`--impl reference` times the float64 CPU oracle on a bounded sample of the same
workload on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "block-scaled GEMM TFLOPS and % of GB300 FP8/FP4 tensor peak, per config"
UNIT = "TFLOPS"
NOMINAL_RATIO = {"mxfp8": 4.5 / 2.25, "nvfp4": 13.5 / 2.25, "bf16": 1.0}  # dense peak vs the bf16 tensor peak
FALLBACK_BF16_TFLOPS = 1900.0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"bf16_tflops": FALLBACK_BF16_TFLOPS, "hbm_gbs": 6800.0}, "fallback"


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() in ("active", "1"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- GPU arm

def _dense_inputs(wl):
    a = wl.a_rows()
    b = wl.b_rows()
    return a, b


def run_ours(args, rank, world, local_rank):
    import torch
    import nvfp4_gemm_moe_gb300 as bsg
    from nvfp4_gemm_moe_gb300 import torch_ops

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = W.ALL[args.workload]
    stream = torch.cuda.current_stream()
    is_dense = isinstance(wl, W.Dense)
    is_dsw = isinstance(wl, W.GroupedDswiglu)
    is_rope = isinstance(wl, W.RopeProj)
    fmt = wl.fmt
    flops = wl.flops

    # ---------------- inputs resident in HBM
    if is_dense:
        a_h, b_h = _dense_inputs(wl)
    elif is_rope:
        a_h, b_h = wl.x_rows()[None], wl.w_rows()[None]
    else:
        a_h, b_h = wl.a_rows()[None], wl.b_rows()
    # bf16 operands are the inputs themselves (the draws rounded to bf16); the others are fp32
    # inputs that every step quantises
    host_dtype = torch.bfloat16 if fmt == "bf16" else torch.float32
    a_pin = torch.from_numpy(a_h).to(host_dtype).pin_memory()
    b_pin = torch.from_numpy(b_h).to(host_dtype).pin_memory()
    del a_h, b_h
    a_d = a_pin.to(dev)
    b_d = b_pin.to(dev)
    la, ma, ka = a_d.shape
    lb, nb, _ = b_d.shape
    if fmt != "bf16":
        v = 32 if fmt == "mxfp8" else 16
        qcols = ka if fmt == "mxfp8" else ka // 2
        qa = torch.empty((la, ma, qcols), dtype=torch.uint8, device=dev)
        qb = torch.empty((lb, nb, qcols), dtype=torch.uint8, device=dev)
        sfa = torch.empty(bsg.bsg_sf_bytes(la, ma, ka, v), dtype=torch.uint8, device=dev)
        sfb = torch.empty(bsg.bsg_sf_bytes(lb, nb, ka, v), dtype=torch.uint8, device=dev)
    ws = torch_ops.new_workspace(dev)
    if is_dense:
        c = torch.empty((wl.l, wl.m, wl.n), dtype=torch.float32 if wl.c_dtype == "f32" else torch.bfloat16,
                        device=dev)
        amax = torch.empty(1, dtype=torch.float32, device=dev)
        outs = None
    elif is_rope:
        cos_h, sin_h = (torch.from_numpy(t).to(torch.bfloat16).pin_memory() for t in wl.tables())
        cos_d, sin_d = cos_h.to(dev), sin_h.to(dev)
        outs = {}
    else:
        offs = torch.from_numpy(wl.padded_offsets()).to(dev)
        alpha = torch.from_numpy(wl.alpha()).to(dev)
        prob = torch.from_numpy(wl.prob()).to(dev)
        nc = torch.ones(1, dtype=torch.float32, device=dev)
        if is_dsw:
            # the stored forward intermediate (valid_m, 2N) in bf16 and the per-expert scale of it
            c_pin = torch.from_numpy(wl.c_rows()).to(torch.bfloat16).pin_memory()
            c_in = c_pin.to(dev)
            beta = torch.from_numpy(wl.beta()).to(dev)
            outs = {"dprob": torch.zeros(wl.valid_m, dtype=torch.float32, device=dev)}
        else:
            outs = {"c": torch.empty((wl.valid_m, wl.n), dtype=torch.bfloat16, device=dev)}

    # the device inputs the step reads (the end-to-end loop alternates two such sets)
    cur = {"a": a_d, "b": b_d}
    if is_rope:
        cur.update(cos=cos_d, sin=sin_d)
    if is_dsw:
        cur.update(c=c_in)

    def gemm():
        if is_dense:
            torch_ops.gemm_amax(qa, qb, sfa, sfb, fmt, wl.m, wl.n, wl.k, wl.l, c=c, amax=amax, workspace=ws)
        elif is_rope and fmt == "bf16":
            outs.update(torch_ops.gemm_rope_bf16(cur["a"][0], cur["b"][0], cur["cos"], cur["sin"], wl.heads,
                                                 wl.head_dim, wl.qk_rope, outputs=outs, workspace=ws))
        elif is_rope:
            outs.update(torch_ops.gemm_rope_mxfp8(qa[0], sfa, qb[0], sfb, cur["cos"], cur["sin"], wl.heads, wl.head_dim,
                                                  wl.qk_rope, outputs=outs, workspace=ws))
        elif is_dsw:
            outs["dprob"].zero_()  # the call adds each row's sum into dprob
            outs.update(torch_ops.grouped_gemm_dswiglu(qa[0], qb, sfa, sfb, fmt, offs, alpha, beta, prob, cur["c"], wl.n,
                                                       wl.k, d_dtype=wl.d_dtype, norm_const=nc, outputs=outs,
                                                       workspace=ws))
        else:
            # the first call allocates D, amax / D_col, SFD_row, SFD_col; later calls reuse them
            outs.update(torch_ops.grouped_gemm_srelu(qa[0], qb, sfa, sfb, fmt, offs, alpha, prob, wl.n, wl.k,
                                                     tanh_clamp_scale=wl.tanh_clamp, d_dtype=wl.d_dtype,
                                                     norm_const=nc, outputs=outs, workspace=ws))

    def step(ev0=None, ev1=None):
        if fmt != "bf16":
            torch_ops.quantize(cur["a"], fmt, q=qa, sf=sfa)
            torch_ops.quantize(cur["b"], fmt, q=qb, sf=sfb)
        if ev0 is not None:
            ev0.record(stream)
        gemm()
        if ev1 is not None:
            ev1.record(stream)

    launches_per_step = 1 if fmt == "bf16" else 3  # (two quantiser kernels +) one GEMM kernel
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if bsg.bsg_read_device_error(ws):
        raise RuntimeError("device error during warm-up")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    g0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    g1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank) if rank == 0 else None
    if clocks:
        clocks.start()
    barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(args.steps):
        step(g0[i], g1[i])
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop() if clocks else None
    elapsed_ms = t0.elapsed_time(t1)
    gemm_ms = [g0[i].elapsed_time(g1[i]) for i in range(args.steps)]
    if bsg.bsg_read_device_error(ws):
        raise RuntimeError("device error in the timed region")

    # ---------------- end to end through the C ABI from pinned host buffers
    # Every step copies its inputs from pinned host memory and reads its results back inside the
    # timed region.  The inputs are double-buffered: step i + 1's host-to-device copies run on a
    # copy stream while step i computes and reads back (the link, not the GPU, bounds this).
    e2e_steps = max(3, min(args.steps, 20))
    names = ["a", "b"] + (["c"] if is_dsw else []) + (["cos", "sin"] if is_rope else [])
    pins = {"a": a_pin, "b": b_pin}
    if is_dsw:
        pins["c"] = c_pin
    if is_rope:
        pins.update(cos=cos_h, sin=sin_h)
    sets = [dict(cur), {k: torch.empty_like(cur[k]) for k in names}]
    if is_dense:
        results = [c, amax]
    elif is_rope:
        results = [outs["out_fp8_row"], outs["out_scales_row"], outs["out_fp8_col"], outs["out_scales_col"]]
    elif is_dsw:
        results = [outs["d_row"], outs["dprob"]] + ([outs["amax"]] if "amax" in outs else [outs["sfd_row"]])
    else:
        results = [outs["c"], outs["d"]] + ([outs["amax"][:1]] if "amax" in outs else [])
    hosts = [torch.empty(r.shape, dtype=r.dtype, pin_memory=True) for r in results]
    h2d = sum(pins[k].numel() * pins[k].element_size() for k in names)
    d2h = sum(r.numel() * r.element_size() for r in results)
    copy_stream = torch.cuda.Stream(device=dev)
    ready = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]

    def copy_in(si):
        copy_stream.wait_event(free[si])  # the step that read this set has finished
        with torch.cuda.stream(copy_stream):
            for k in names:
                sets[si][k].copy_(pins[k], non_blocking=True)
        ready[si].record(copy_stream)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    copy_stream.wait_event(e0)
    copy_in(0)
    for i in range(e2e_steps):
        si = i % 2
        if i + 1 < e2e_steps:
            copy_in(1 - si)
        stream.wait_event(ready[si])
        cur.update(sets[si])
        step()
        free[si].record(stream)
        for h, r in zip(hosts, results):
            h.copy_(r, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    cur.update(sets[0])
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    # ---------------- max over ranks
    elapsed_ms, e2e_ms, gemm_mean_ms = max_over_ranks([elapsed_ms, e2e_ms, statistics.mean(gemm_ms)], world, dev)
    ms_per_step = elapsed_ms / args.steps
    value = replica_throughput(flops * args.steps, elapsed_ms, world)
    e2e_value = replica_throughput(flops, e2e_ms, world)

    peaks, peak_src = load_peaks()
    peak = peaks["bf16_tflops"] * NOMINAL_RATIO[fmt]
    achieved = flops / (gemm_mean_ms * 1e-3) / 1e12
    roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "traffic": _traffic(args.workload),
            "kernel": "GEMM launch (automatic choice: gemm_pair_kernel or gemm_kernel)", "peak_source": f"{peak_src} bf16 burst x {NOMINAL_RATIO[fmt]:g} "
                                                   f"(dense {fmt} / bf16 nominal ratio)"}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {"mxfp8": "e4m3", "nvfp4": "e2m1", "bf16": "bf16"}[fmt], "data": "synthetic",
        "config": _config(wl),
        "roofline": roof,
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 3)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "gemm_ms": round(gemm_mean_ms, 4),
    }
    if args.per_config and world == 1 and args.workload == W.DENSE_MXFP8_8192.name:
        line["per_config"] = per_config_records(dev, peaks, peak_src)
    return line


# --------------------------------------------------------------------------- per-config GEMM records

# The other workloads the metric is quoted per config on, measured in the default run beside the
# headline: (label, workload, C present).  The E4M3-D workload is also timed with C = NULL (C is
# an optional output of the grouped operation).
PER_CONFIG = (
    ("1", W.DENSE_MXFP8_256.name, True),
    ("3", W.DENSE_NVFP4_16384.name, True),
    ("4", W.GROUPED_SRELU_E32.name, True),
    ("4'", W.GROUPED_SRELU_E32_CLAMP.name, True),
    ("5", W.GROUPED_FP8D_E128.name, True),
    ("5 (C = NULL)", W.GROUPED_FP8D_E128.name, False),
)
PER_CONFIG_REGION_S = 0.25  # each config's timed region lasts at least this long (clock samples)


def _dense_bytes(wl):
    """Algorithmic HBM bytes of one dense GEMM launch: codes and scales of A and B once, C once."""
    per_elem = 1.0 if wl.fmt == "mxfp8" else 0.5
    ab = wl.l * (wl.m + wl.n) * wl.k * (per_elem + 1.0 / wl.sf_vec)
    c = wl.l * wl.m * wl.n * (4 if wl.c_dtype == "f32" else 2)
    return ab + c + 4


def per_config_records(dev, peaks, peak_src, entries=PER_CONFIG):
    """GEMM launch time (CUDA events around back-to-back launches on the current stream, inputs
    quantised once beforehand), TFLOP/s, fraction of the FP8 / FP4 peak, traffic and clocks for
    every per-config workload."""
    import torch
    from nvfp4_gemm_moe_gb300 import torch_ops
    stream = torch.cuda.current_stream()
    recs = []
    cache = {}
    for label, name, with_c in entries:
        wl = W.ALL[name]
        # the clamp variant and the C = NULL run reuse the operands of the workload before them
        key = name if isinstance(wl, W.Dense) else (wl.experts, wl.k, wl.n, wl.routed_rows, wl.skew, wl.seed, wl.fmt)
        if key not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            if isinstance(wl, W.Dense):
                a, b = wl.a_rows(), wl.b_rows()
            else:
                a, b = wl.a_rows()[None], wl.b_rows()
            a_d = torch.from_numpy(a).to(dev)
            del a
            qa, sfa = torch_ops.quantize(a_d, wl.fmt)
            del a_d
            b_d = torch.from_numpy(b).to(dev)
            del b
            qb, sfb = torch_ops.quantize(b_d, wl.fmt)
            del b_d
            cache[key] = (qa, sfa, qb, sfb)
        qa, sfa, qb, sfb = cache[key]
        ws = torch_ops.new_workspace(dev)
        if isinstance(wl, W.Dense):
            c = torch.empty((wl.l, wl.m, wl.n), dtype=torch.float32 if wl.c_dtype == "f32" else torch.bfloat16,
                            device=dev)
            amax = torch.empty(1, dtype=torch.float32, device=dev)

            def call():
                torch_ops.gemm_amax(qa, qb, sfa, sfb, wl.fmt, wl.m, wl.n, wl.k, wl.l, c=c, amax=amax, workspace=ws)
        else:
            offs = torch.from_numpy(wl.padded_offsets()).to(dev)
            alpha = torch.from_numpy(wl.alpha()).to(dev)
            prob = torch.from_numpy(wl.prob()).to(dev)
            nc = torch.ones(1, dtype=torch.float32, device=dev)
            outs = torch_ops.grouped_gemm_srelu(qa[0], qb, sfa, sfb, wl.fmt, offs, alpha, prob, wl.n, wl.k,
                                                tanh_clamp_scale=wl.tanh_clamp, d_dtype=wl.d_dtype, norm_const=nc,
                                                c_dtype=torch.bfloat16 if with_c else None, workspace=ws)

            def call():
                torch_ops.grouped_gemm_srelu(qa[0], qb, sfa, sfb, wl.fmt, offs, alpha, prob, wl.n, wl.k,
                                             tanh_clamp_scale=wl.tanh_clamp, d_dtype=wl.d_dtype, norm_const=nc,
                                             outputs=outs, workspace=ws)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        t = time.perf_counter()
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        est = max((time.perf_counter() - t) / 3, 1e-6)
        calls = int(max(20, min(20000, PER_CONFIG_REGION_S / est)))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clocks = ClockSampler(dev.index or 0)
        clocks.start()
        e0.record(stream)
        for _ in range(calls):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
        clk = clocks.stop()
        import nvfp4_gemm_moe_gb300 as bsg
        if bsg.bsg_read_device_error(ws):
            raise RuntimeError(f"device error in the per-config run of {name}")
        ms = e0.elapsed_time(e1) / calls
        peak = peaks["bf16_tflops"] * NOMINAL_RATIO[wl.fmt]
        tf = wl.flops / (ms * 1e-3) / 1e12
        rec = {"config": label, "workload": name, "format": wl.fmt, "calls": calls, "gemm_ms": round(ms, 5),
               "tflops": round(tf, 1), "peak": round(peak, 1), "frac": round(tf / peak, 4),
               "peak_source": f"{peak_src} bf16 burst x {NOMINAL_RATIO[wl.fmt]:g}",
               "traffic": _traffic(name) if with_c else None, "clocks": clk}
        if isinstance(wl, W.Dense):
            gb = _dense_bytes(wl)
            rec.update(flops=wl.flops, algorithmic_bytes=int(gb), gbs=round(gb / (ms * 1e-3) / 1e9, 1),
                       l2="inputs and outputs stay in L2 between calls" if gb < 64e6 else
                       "no flush: C written per call exceeds L2")
        else:
            useful = 2.0 * wl.routed_rows * wl.n * wl.k
            rec.update(flops=wl.flops, valid_m=wl.valid_m, routed_rows=wl.routed_rows,
                       useful_tflops=round(useful / (ms * 1e-3) / 1e12, 1),
                       useful_note="2 * routed_rows * N * K (padding rows excluded)",
                       c=("bf16" if with_c else None), d_dtype=wl.d_dtype, tanh_clamp=wl.tanh_clamp,
                       l2="no flush: operands and outputs exceed L2")
        if label == "1":
            rec.update(_latency_graph(call, stream))
        recs.append(rec)
    cache.clear()
    torch.cuda.empty_cache()
    return recs


def _latency_graph(call, stream, per_graph=100, replays=20):
    """Per-call device time of a launch-bound call: `per_graph` calls captured into one CUDA graph,
    replayed `replays` times between CUDA events (no host work between the calls)."""
    import torch
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(stream)
    with torch.cuda.stream(s):
        call()  # an eager call on the capture stream first (per-device set-up happens outside capture)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            for _ in range(per_graph):
                call()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(replays):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (per_graph * replays)
    return {"us_per_call_graph": round(us, 2), "graph_calls": per_graph * replays}


def max_over_ranks(times_ms, world, device="cpu"):
    """Each time maximised over the ranks (every rank gets the result); identity for one rank."""
    import torch
    if world <= 1:
        return [float(t) for t in times_ms]
    import torch.distributed as dist
    t = torch.tensor([float(x) for x in times_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def replica_throughput(flops_per_rank, elapsed_ms, world):
    """TFLOP/s of the whole job: every rank ran the same work in at most elapsed_ms."""
    return world * flops_per_rank / (elapsed_ms * 1e-3) / 1e12


def _traffic(workload):
    """DRAM bytes per GEMM launch from the committed ncu summary, if one exists for this workload."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get(workload)
    return None


def _config(wl):
    if isinstance(wl, W.RopeProj) and wl.fmt == "bf16":
        out_gb = 2 * wl.tokens * wl.n / 1e9
        return {"workload": wl.name, "format": wl.fmt, "tokens": wl.tokens, "q_lora": wl.q_lora, "heads": wl.heads,
                "head_dim": wl.head_dim, "qk_rope": wl.qk_rope, "flops_per_step": wl.flops,
                "l2": "no explicit flush: each step writes %.2f GB of outputs, more than L2, after reading its "
                      "%.2f GB of bf16 inputs" % (out_gb, (wl.tokens + wl.n) * wl.q_lora * 2 / 1e9),
                "step": "projection GEMM/RoPE/row+column MXFP8 on bf16 x and w"}
    if isinstance(wl, W.RopeProj):
        return {"workload": wl.name, "format": wl.fmt, "tokens": wl.tokens, "q_lora": wl.q_lora, "heads": wl.heads,
                "head_dim": wl.head_dim, "qk_rope": wl.qk_rope, "flops_per_step": wl.flops,
                "l2": "no flush: fp32 inputs of %.2f GB exceed L2" % ((wl.tokens + wl.n) * wl.q_lora * 4 / 1e9),
                "step": "quantise x + quantise w + projection GEMM/RoPE/row+column MXFP8"}
    if isinstance(wl, W.Dense):
        return {"workload": wl.name, "format": wl.fmt, "m": wl.m, "n": wl.n, "k": wl.k, "l": wl.l,
                "c_dtype": wl.c_dtype, "flops_per_step": wl.flops,
                "l2": "no flush: fp32 inputs of 2 x %.2f GB exceed L2" % (wl.l * wl.m * wl.k * 4 / 1e9),
                "step": "quantise A + quantise B + GEMM/amax"}
    if isinstance(wl, W.GroupedDswiglu):
        return {"workload": wl.name, "format": wl.fmt, "experts": wl.experts, "n": wl.n, "k": wl.k,
                "valid_m": wl.valid_m, "routed_rows": wl.routed_rows, "c_dtype": wl.c_dtype, "d_dtype": wl.d_dtype,
                "flops_per_step": wl.flops, "l2": "no flush: fp32 inputs exceed L2",
                "step": "quantise A + quantise B + grouped GEMM/dSwiGLU backward (C read, D and dprob written)"}
    return {"workload": wl.name, "format": wl.fmt, "experts": wl.experts, "n": wl.n, "k": wl.k,
            "valid_m": wl.valid_m, "routed_rows": wl.routed_rows, "d_dtype": wl.d_dtype, "tanh_clamp": wl.tanh_clamp,
            "flops_per_step": wl.flops, "l2": "no flush: fp32 inputs exceed L2",
            "step": "quantise A + quantise B + grouped GEMM/sReLU"}


# --------------------------------------------------------------------------- reference arm (CPU oracle)

ORACLE_SAMPLE_FLOPS = 6e11  # float64 GEMM work of one oracle sample (about 10-30 s on the host cores)


def oracle_rows(wl, requested=0):
    """Rows of A in the oracle's timed sample: `requested`, else enough for ORACLE_SAMPLE_FLOPS."""
    if requested > 0:
        return int(requested)
    if isinstance(wl, W.RopeProj):
        return max(256, min(int(ORACLE_SAMPLE_FLOPS / (2.0 * wl.n * wl.q_lora)) // 256 * 256, wl.tokens))
    max_rows = wl.m if isinstance(wl, W.Dense) else wl.valid_m
    rows = int(ORACLE_SAMPLE_FLOPS / (2.0 * wl.n * wl.k)) // 256 * 256
    return max(256, min(rows, max_rows))


def run_reference(args):
    from oracle import dswiglu as od, gemm as og, quantize as oq, rope as orope
    wl = W.ALL[args.workload]
    cores = os.cpu_count() or 1
    step_times, sample_flops = [], 0.0
    args.ref_rows = oracle_rows(wl, args.ref_rows)

    def one_step():
        if isinstance(wl, W.RopeProj) and wl.fmt == "bf16":
            import torch
            rows = np.arange(args.ref_rows)            # the first tokens, all heads
            xb = torch.from_numpy(wl.x_rows(rows)).to(torch.bfloat16).double().numpy()
            wb = torch.from_numpy(wl.w_rows()).to(torch.bfloat16).double().numpy()
            cos, sin = (torch.from_numpy(t[:len(rows)]).to(torch.bfloat16).double().numpy() for t in wl.tables())
            orope.project_bf16(xb, wb, cos, sin, wl.heads, wl.head_dim, wl.qk_rope)
            return 2.0 * len(rows) * wl.n * wl.q_lora
        if isinstance(wl, W.RopeProj):
            rows = np.arange(args.ref_rows)            # the first tokens, all heads
            xc, xs = oq.quantize_logical(wl.x_rows(rows)[None], wl.fmt)
            wc, wsc = oq.quantize_logical(wl.w_rows()[None], wl.fmt)
            cos, sin = (t[:len(rows)] for t in wl.tables())
            orope.project(xc[0], xs[0], wc[0], wsc[0], cos, sin, wl.heads, wl.head_dim, wl.qk_rope)
            return 2.0 * len(rows) * wl.n * wl.q_lora
        if isinstance(wl, W.Dense):
            rows = np.arange(args.ref_rows)           # first rows of batch 0 of A
            a = wl.a_rows(rows)[None]
            b = wl.b_rows(np.arange(wl.n))[None]       # all of B for batch 0
            qa, sfa = oq.quantize(a, wl.fmt)
            qb, sfb = oq.quantize(b, wl.fmt)
            c, amax = og.dense_gemm_amax(qa, qb, sfa, sfb, wl.fmt, len(rows), wl.n, wl.k, 1)
            return 2.0 * len(rows) * wl.n * wl.k
        offs = wl.padded_offsets()
        rows = np.arange(args.ref_rows)
        g = 0
        a = wl.a_rows(rows)[None]
        b = wl.b_rows(np.arange(wl.n))[None]  # expert 0's weights
        qa, sfa = oq.quantize(a, wl.fmt)
        qb, sfb = oq.quantize(b, wl.fmt)
        o = np.array([len(rows)], np.int32)
        if isinstance(wl, W.GroupedDswiglu):
            c_vals = wl.c_rows(rows)  # fp32 draws; the GPU arm stores them as bf16
            od.grouped_dswiglu(qa[0], qb, sfa, sfb, wl.fmt, o, wl.alpha()[:1], wl.beta()[:1], wl.prob()[:len(rows)],
                               c_vals, wl.k, wl.n, d_fp8=(wl.d_dtype == "e4m3"))
            return 2.0 * len(rows) * wl.n * wl.k
        og.grouped_srelu(qa[0], qb, sfa, sfb, wl.fmt, o, wl.alpha()[:1], wl.prob()[:len(rows)], wl.k, wl.n,
                         tanh_clamp_scale=wl.tanh_clamp, d_fp8=(wl.d_dtype == "e4m3"))
        del g, offs
        return 2.0 * len(rows) * wl.n * wl.k

    for _ in range(args.warmup):
        one_step()
    for _ in range(args.steps):
        t = time.perf_counter()
        sample_flops = one_step()
        step_times.append(time.perf_counter() - t)
    total = sum(step_times)
    value = sample_flops * args.steps / total / 1e12
    steps_txt = ("float64 GEMM on the bf16 values, epilogue" if wl.fmt == "bf16"
                 else "quantise, dequantise, float64 GEMM, epilogue")
    sample = (f"oracle path ({steps_txt}) on the first {args.ref_rows} rows of A "
              f"against all {wl.n} rows of B (batch/expert 0) of {wl.name}; numpy/BLAS float64 on {cores} host threads")
    line = {
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": _config(wl),
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def cpu_baseline(args):
    """The oracle timed on a bounded sample (about 10-30 s of host work) for the GPU arm's line."""
    class A:
        pass
    ra = A()
    ra.workload, ra.steps, ra.warmup, ra.ref_rows = args.workload, 1, 0, args.ref_rows
    t = time.perf_counter()
    line = run_reference(ra)
    cb = line["cpu_baseline"]
    cb["wall_s"] = round(time.perf_counter() - t, 2)
    return cb


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=W.DENSE_MXFP8_8192.name, choices=sorted(W.ALL))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-rows", type=int, default=0,
                    help="rows of A in the oracle's timed sample (0: sized to about 6e11 float64 flops)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="skip the GEMM records of the other configs (measured by default at N = 1)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            if args.steps > 3:
                args.steps = 3  # each oracle step is a bounded host sample of several seconds
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

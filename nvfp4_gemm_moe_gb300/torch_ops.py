"""Torch-facing helpers: allocate output tensors with torch and call the C ABI.

PyTorch supplies device memory and the stream only; the arithmetic runs in the
library's kernels through the binding functions of this package.
"""
from __future__ import annotations

import torch

from . import (BF16, E2M1, E4M3, F16, F32, FORMATS, bsg_gemm_amax, bsg_gemm_rope_bf16, bsg_gemm_rope_mxfp8,
               bsg_grouped_discrete_workspace_size, bsg_grouped_gemm_dswiglu, bsg_grouped_gemm_srelu,
               bsg_grouped_gemm_srelu_discrete, bsg_quantize_mx, bsg_quantize_mx_bf16, bsg_rope_workspace_size,
               bsg_sf_bytes, bsg_workspace_size)


def new_workspace(device="cuda") -> torch.Tensor:
    return torch.zeros(bsg_workspace_size(), dtype=torch.uint8, device=device)


def quantize(x: torch.Tensor, fmt: str, q=None, sf=None, stream=None):
    """x: fp32 or bf16 (batch, rows, K) or (rows, K) on the GPU -> (codes uint8, sf uint8 flat)."""
    if x.dim() == 2:
        x = x.unsqueeze(0)
    batch, rows, k = x.shape
    ab, sfd, v = FORMATS[fmt]
    q_cols = k if fmt == "mxfp8" else k // 2
    if q is None:
        q = torch.empty((batch, rows, q_cols), dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty(bsg_sf_bytes(batch, rows, k, v), dtype=torch.uint8, device=x.device)
    if x.dtype == torch.bfloat16:
        bsg_quantize_mx_bf16(x, batch, rows, k, ab, v, sfd, q, sf, stream=stream)
    elif x.dtype == torch.float32:
        bsg_quantize_mx(x, batch, rows, k, ab, v, sfd, q, sf, stream=stream)
    else:
        raise TypeError(f"quantize takes fp32 or bf16 input, not {x.dtype}")
    return q, sf


# C / D element types: torch dtypes, or "e4m3" / "e2m1" for plain FP8 / packed FP4 outputs (uint8 tensors)
_OUT_KINDS = {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16, "e4m3": E4M3, "e2m1": E2M1,
              "f32": F32, "bf16": BF16, "f16": F16}
_TORCH_OUT = {F32: torch.float32, BF16: torch.bfloat16, F16: torch.float16}


def _out_tensor(kind, rows, n, lead, dev):
    shape = (lead, rows, n) if lead is not None else (rows, n)
    if kind in _TORCH_OUT:
        return torch.empty(shape, dtype=_TORCH_OUT[kind], device=dev)
    cols = n if kind == E4M3 else n // 2
    return torch.empty(shape[:-1] + (cols,), dtype=torch.uint8, device=dev)


def gemm_amax(a, b, sfa, sfb, fmt: str, m: int, n: int, k: int, l: int, c_dtype=torch.bfloat16, c=None,
              amax=None, workspace=None, stream=None, **opts):
    """C (l, m, n) of c_dtype (torch.float32 / bfloat16 / float16, or "e4m3" / "e2m1" with NVFP4
    operands, returned as uint8) and the fp32 amax."""
    ab, sfd, v = FORMATS[fmt]
    dev = a.device
    ck = _OUT_KINDS[c_dtype] if c is None or c.dtype == torch.uint8 else _OUT_KINDS[c.dtype]
    if c is None:
        c = _out_tensor(ck, m, n, l, dev)
    if amax is None:
        amax = torch.empty(1, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_workspace(dev)
    bsg_gemm_amax(a, b, sfa, sfb, ab, sfd, v, m, n, k, l, c, ck, amax, workspace, stream=stream, **opts)
    return c, amax


def _grouped_outputs(valid_m, n, num_experts, d_dtype, c_dtype, norm_const, outputs, dev):
    out = dict(outputs or {})
    if "c" not in out:
        out["c"] = None if c_dtype is None else torch.empty((valid_m, n), dtype=c_dtype, device=dev)
    if d_dtype in ("bf16", "f16", "f32"):
        dk = _OUT_KINDS[d_dtype]
        out.setdefault("d", _out_tensor(dk, valid_m, n, None, dev))
        out.setdefault("amax", torch.empty(num_experts, dtype=torch.float32, device=dev))
    else:
        out.setdefault("d", torch.empty((valid_m, n), dtype=torch.uint8, device=dev))
        out.setdefault("d_col", torch.empty((valid_m, n), dtype=torch.uint8, device=dev))
        out.setdefault("sfd_row", torch.empty(bsg_sf_bytes(1, valid_m, n, 32), dtype=torch.uint8, device=dev))
        out.setdefault("sfd_col", torch.empty(bsg_sf_bytes(1, n, valid_m, 32), dtype=torch.uint8, device=dev))
        if norm_const is None:
            norm_const = torch.ones(1, dtype=torch.float32, device=dev)
        dk = E4M3
    c = out["c"]
    ck = BF16 if c is None else _OUT_KINDS[c.dtype]
    return out, dk, ck, norm_const


def grouped_gemm_srelu(a, b, sfa, sfb, fmt: str, padded_offsets, alpha, prob, n: int, k: int,
                       tanh_clamp_scale=None, d_dtype="bf16", c_dtype=torch.bfloat16, norm_const=None,
                       outputs=None, workspace=None, stream=None, **opts):
    """Returns a dict of the outputs (c, d, amax or d, d_col, sfd_row, sfd_col); d_dtype is
    "bf16", "f16", "f32" or "e4m3", c_dtype a torch float dtype or None."""
    ab, sfd, v = FORMATS[fmt]
    dev = a.device
    valid_m = a.shape[0] if a.dim() == 2 else a.shape[1]
    num_experts = padded_offsets.numel()
    out, dk, ck, norm_const = _grouped_outputs(valid_m, n, num_experts, d_dtype, c_dtype, norm_const, outputs, dev)
    if workspace is None:
        workspace = new_workspace(dev)
    bsg_grouped_gemm_srelu(a, b, sfa, sfb, ab, sfd, v, valid_m, n, k, num_experts, padded_offsets, alpha, prob,
                           tanh_clamp_scale, norm_const, out["c"], ck, out["d"], out.get("d_col"), dk,
                           out.get("sfd_row"), out.get("sfd_col"), out.get("amax"), workspace, stream=stream, **opts)
    return out


def _pointer_array(ptrs, dev):
    if isinstance(ptrs, torch.Tensor):
        return ptrs
    return torch.tensor([t.data_ptr() for t in ptrs], dtype=torch.int64, device=dev)


def grouped_gemm_srelu_discrete(a, b_ptrs, sfa, sfb_ptrs, fmt: str, padded_offsets, alpha, prob, n: int, k: int,
                                tanh_clamp_scale=None, d_dtype="bf16", c_dtype=torch.bfloat16, norm_const=None,
                                outputs=None, workspace=None, stream=None, **opts):
    """grouped_gemm_srelu with per-expert weights: b_ptrs / sfb_ptrs are lists of the experts'
    code tensors (n, k) / SF buffers, or device int64 tensors of their addresses.  The experts'
    TMA descriptors are built on the device (no synchronisation; the call can be captured in a
    CUDA graph); invalid addresses show up as BSG_DEVERR_BAD_POINTERS."""
    ab, sfd, v = FORMATS[fmt]
    dev = a.device
    valid_m = a.shape[0] if a.dim() == 2 else a.shape[1]
    num_experts = padded_offsets.numel()
    bp, sp = _pointer_array(b_ptrs, dev), _pointer_array(sfb_ptrs, dev)
    out, dk, ck, norm_const = _grouped_outputs(valid_m, n, num_experts, d_dtype, c_dtype, norm_const, outputs, dev)
    if workspace is None:
        workspace = torch.zeros(bsg_grouped_discrete_workspace_size(num_experts), dtype=torch.uint8, device=dev)
    bsg_grouped_gemm_srelu_discrete(a, bp, sfa, sp, ab, sfd, v, valid_m, n, k, num_experts, padded_offsets, alpha,
                                    prob, tanh_clamp_scale, norm_const, out["c"], ck, out["d"], out.get("d_col"), dk,
                                    out.get("sfd_row"), out.get("sfd_col"), out.get("amax"), workspace,
                                    stream=stream, **opts)
    return out


def grouped_gemm_dswiglu(a, b, sfa, sfb, fmt: str, padded_offsets, alpha, beta, prob, c, n: int, k: int,
                         c_dtype=None, d_dtype="bf16", norm_const=None, outputs=None, workspace=None, stream=None,
                         **opts):
    """dSwiGLU backward over the grouped GEMM.  ``c`` (valid_m, 2n) is the stored forward
    intermediate (a bf16 / f16 / f32 tensor, or uint8 E4M3 codes with c_dtype="e4m3").  Returns a
    dict: d_row, dprob (fresh zeros unless given: the call adds into it) and amax (L, 2) for
    d_dtype "bf16" / "f16" / "f32", or d_row, d_col, sfd_row, sfd_col and dprob for "e4m3"."""
    ab, sfd, v = FORMATS[fmt]
    dev = a.device
    valid_m = a.shape[0] if a.dim() == 2 else a.shape[1]
    num_experts = padded_offsets.numel()
    ck = _OUT_KINDS[c_dtype] if c_dtype is not None else _OUT_KINDS[c.dtype]
    out = dict(outputs or {})
    out.setdefault("dprob", torch.zeros(valid_m, dtype=torch.float32, device=dev))
    if d_dtype in ("bf16", "f16", "f32"):
        dk = _OUT_KINDS[d_dtype]
        out.setdefault("d_row", _out_tensor(dk, valid_m, 2 * n, None, dev))
        out.setdefault("amax", torch.empty((num_experts, 2), dtype=torch.float32, device=dev))
    else:
        dk = E4M3
        out.setdefault("d_row", torch.empty((valid_m, 2 * n), dtype=torch.uint8, device=dev))
        out.setdefault("d_col", torch.empty((valid_m, 2 * n), dtype=torch.uint8, device=dev))
        out.setdefault("sfd_row", torch.empty(bsg_sf_bytes(1, valid_m, 2 * n, 32), dtype=torch.uint8, device=dev))
        out.setdefault("sfd_col", torch.empty(bsg_sf_bytes(1, 2 * n, valid_m, 32), dtype=torch.uint8, device=dev))
        if norm_const is None:
            norm_const = torch.ones(1, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_workspace(dev)
    bsg_grouped_gemm_dswiglu(a, b, sfa, sfb, ab, sfd, v, valid_m, n, k, num_experts, padded_offsets, alpha, beta,
                             prob, c, ck, norm_const, out["d_row"], out.get("d_col"), dk, out.get("sfd_row"),
                             out.get("sfd_col"), out["dprob"], out.get("amax"), workspace, stream=stream, **opts)
    return out


def gemm_rope_mxfp8(x, x_scale, w, w_scale, cos, sin, num_heads: int, head_dim: int = 192, qk_rope: int = 64,
                    scale_layout: str = "atoms", outputs=None, workspace=None, stream=None, **opts):
    """Projection GEMM + per-head RoPE + row / column MXFP8.  x (tokens, q_lora) and w
    (num_heads * head_dim, q_lora) are E4M3 codes (uint8); x_scale / w_scale their E8M0 scales,
    in the atom layout of ``quantize`` (scale_layout="atoms") or plain (rows, q_lora / 32)
    ("plain"); cos / sin bf16 (tokens, qk_rope).  Returns a dict: out_fp8_row, out_scales_row,
    out_fp8_col, out_scales_col."""
    tokens, q_lora = x.shape[-2], x.shape[-1]
    dev = x.device
    out = dict(outputs or {})
    out.setdefault("out_fp8_row", torch.empty((tokens, num_heads, head_dim), dtype=torch.uint8, device=dev))
    out.setdefault("out_scales_row", torch.empty((tokens, num_heads, head_dim // 32), dtype=torch.uint8, device=dev))
    out.setdefault("out_fp8_col", torch.empty((tokens, num_heads, head_dim), dtype=torch.uint8, device=dev))
    out.setdefault("out_scales_col", torch.empty((tokens // 32, num_heads, head_dim), dtype=torch.uint8, device=dev))
    layout = {"atoms": 0, "plain": 1}[scale_layout]
    if workspace is None:
        workspace = torch.zeros(bsg_rope_workspace_size(tokens, num_heads, head_dim, q_lora), dtype=torch.uint8,
                                device=dev)
    bsg_gemm_rope_mxfp8(x, x_scale, w, w_scale, layout, cos, sin, tokens, q_lora, num_heads, head_dim, qk_rope,
                        out["out_fp8_row"], out["out_scales_row"], out["out_fp8_col"], out["out_scales_col"],
                        workspace, workspace_bytes=workspace.numel(), stream=stream, **opts)
    return out


def gemm_rope_bf16(x, w, cos, sin, num_heads: int, head_dim: int = 192, qk_rope: int = 64, outputs=None,
                   workspace=None, stream=None, **opts):
    """The BF16-input projection: x (tokens, q_lora) and w (num_heads * head_dim, q_lora) bf16,
    K-major; the rest (RoPE, dual MXFP8 outputs) as ``gemm_rope_mxfp8``."""
    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16:
        raise TypeError("gemm_rope_bf16 takes bf16 x and w")
    tokens, q_lora = x.shape[-2], x.shape[-1]
    dev = x.device
    out = dict(outputs or {})
    out.setdefault("out_fp8_row", torch.empty((tokens, num_heads, head_dim), dtype=torch.uint8, device=dev))
    out.setdefault("out_scales_row", torch.empty((tokens, num_heads, head_dim // 32), dtype=torch.uint8, device=dev))
    out.setdefault("out_fp8_col", torch.empty((tokens, num_heads, head_dim), dtype=torch.uint8, device=dev))
    out.setdefault("out_scales_col", torch.empty((tokens // 32, num_heads, head_dim), dtype=torch.uint8, device=dev))
    if workspace is None:
        workspace = torch.zeros(bsg_workspace_size(), dtype=torch.uint8, device=dev)
    bsg_gemm_rope_bf16(x, w, cos, sin, tokens, q_lora, num_heads, head_dim, qk_rope, out["out_fp8_row"],
                       out["out_scales_row"], out["out_fp8_col"], out["out_scales_col"], workspace,
                       workspace_bytes=workspace.numel(), stream=stream, **opts)
    return out

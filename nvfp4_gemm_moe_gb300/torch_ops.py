"""Torch-facing helpers: allocate output tensors with torch and call the C ABI.

PyTorch supplies device memory and the stream only; the arithmetic runs in the
library's kernels through the binding functions of this package.
"""
from __future__ import annotations

import torch

from . import (BF16, E4M3, F32, FORMATS, bsg_gemm_amax, bsg_grouped_gemm_srelu, bsg_quantize_mx, bsg_sf_bytes,
               bsg_workspace_size)


def new_workspace(device="cuda") -> torch.Tensor:
    return torch.zeros(bsg_workspace_size(), dtype=torch.uint8, device=device)


def quantize(x: torch.Tensor, fmt: str, q=None, sf=None, stream=None):
    """x: fp32 (batch, rows, K) or (rows, K) on the GPU -> (codes uint8, sf uint8 flat)."""
    if x.dim() == 2:
        x = x.unsqueeze(0)
    batch, rows, k = x.shape
    ab, sfd, v = FORMATS[fmt]
    q_cols = k if fmt == "mxfp8" else k // 2
    if q is None:
        q = torch.empty((batch, rows, q_cols), dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty(bsg_sf_bytes(batch, rows, k, v), dtype=torch.uint8, device=x.device)
    bsg_quantize_mx(x, batch, rows, k, ab, v, sfd, q, sf, stream=stream)
    return q, sf


def gemm_amax(a, b, sfa, sfb, fmt: str, m: int, n: int, k: int, l: int, c_dtype=torch.bfloat16, c=None,
              amax=None, workspace=None, stream=None, **opts):
    ab, sfd, v = FORMATS[fmt]
    dev = a.device
    if c is None:
        c = torch.empty((l, m, n), dtype=c_dtype, device=dev)
    if amax is None:
        amax = torch.empty(1, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_workspace(dev)
    ck = F32 if c.dtype == torch.float32 else BF16
    bsg_gemm_amax(a, b, sfa, sfb, ab, sfd, v, m, n, k, l, c, ck, amax, workspace, stream=stream, **opts)
    return c, amax


def grouped_gemm_srelu(a, b, sfa, sfb, fmt: str, padded_offsets, alpha, prob, n: int, k: int,
                       tanh_clamp_scale=None, d_dtype="bf16", c_dtype=torch.bfloat16, norm_const=None,
                       outputs=None, workspace=None, stream=None, **opts):
    """Returns a dict of the outputs (c, d, amax or d, d_col, sfd_row, sfd_col)."""
    ab, sfd, v = FORMATS[fmt]
    dev = a.device
    valid_m = a.shape[0] if a.dim() == 2 else a.shape[1]
    num_experts = padded_offsets.numel()
    out = dict(outputs or {})
    if "c" not in out:
        out["c"] = None if c_dtype is None else torch.empty((valid_m, n), dtype=c_dtype, device=dev)
    if d_dtype == "bf16":
        out.setdefault("d", torch.empty((valid_m, n), dtype=torch.bfloat16, device=dev))
        out.setdefault("amax", torch.empty(num_experts, dtype=torch.float32, device=dev))
        dk = BF16
    else:
        out.setdefault("d", torch.empty((valid_m, n), dtype=torch.uint8, device=dev))
        out.setdefault("d_col", torch.empty((valid_m, n), dtype=torch.uint8, device=dev))
        out.setdefault("sfd_row", torch.empty(bsg_sf_bytes(1, valid_m, n, 32), dtype=torch.uint8, device=dev))
        out.setdefault("sfd_col", torch.empty(bsg_sf_bytes(1, n, valid_m, 32), dtype=torch.uint8, device=dev))
        if norm_const is None:
            norm_const = torch.ones(1, dtype=torch.float32, device=dev)
        dk = E4M3
    if workspace is None:
        workspace = new_workspace(dev)
    c = out["c"]
    ck = BF16 if c is None or c.dtype == torch.bfloat16 else F32
    bsg_grouped_gemm_srelu(a, b, sfa, sfb, ab, sfd, v, valid_m, n, k, num_experts, padded_offsets, alpha, prob,
                           tanh_clamp_scale, norm_const, c, ck, out["d"], out.get("d_col"), dk, out.get("sfd_row"),
                           out.get("sfd_col"), out.get("amax"), workspace, stream=stream, **opts)
    return out

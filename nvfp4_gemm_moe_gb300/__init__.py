"""Python binding of the block-scaled GEMM C ABI (``include/bsg.h``).

Argument marshalling only: every function here converts its arguments (torch
tensors or raw integer device pointers, enums, the current torch stream) and
calls the entry point of the same name in ``libbsg.so``; all computation runs in
the library's CUDA kernels.  There is no fallback: importing this package
without the built library raises, and a non-OK status raises ``BsgError``.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build_mod

# dtype / status enums (bsg.h)
E4M3, E5M2, E2M1, F32, BF16, F16 = 0, 1, 2, 3, 4, 5
SF_UE8M0, SF_UE4M3 = 0, 1
OK = 0
DEVERR_TIMEOUT, DEVERR_BAD_OFFSETS, DEVERR_BAD_POINTERS = 0x1, 0x2, 0x4

MXFP8 = (E4M3, SF_UE8M0, 32)
NVFP4 = (E2M1, SF_UE4M3, 16)
FORMATS = {"mxfp8": MXFP8, "nvfp4": NVFP4}

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "bsg.h")


class BsgError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_lib.bsg_status_string(status).decode()} ({status})")


class bsg_gemm_opts(ctypes.Structure):
    _fields_ = [("tile_n", ctypes.c_int), ("max_ctas", ctypes.c_int), ("tanh_approx", ctypes.c_int),
                ("validate_offsets", ctypes.c_int), ("cta_pair", ctypes.c_int), ("b_major", ctypes.c_int),
                ("reserved", ctypes.c_int * 2)]


def _load():
    # BSG_LIBRARY names a prebuilt library file to load instead of the in-tree build
    path = os.environ.get("BSG_LIBRARY") or _build_mod.LIB
    if not os.environ.get("BSG_LIBRARY") and (not os.path.exists(path) or
                                              os.environ.get("BSG_AUTOBUILD", "1") == "1"):
        path = _build_mod.build()
    lib = ctypes.CDLL(path)
    P, I64, I, F, SZ, U32P = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t,
                              ctypes.POINTER(ctypes.c_uint32))
    lib.bsg_workspace_size.restype = SZ
    lib.bsg_workspace_size.argtypes = []
    lib.bsg_sf_bytes.restype = SZ
    lib.bsg_sf_bytes.argtypes = [I64, I64, I64, I]
    lib.bsg_status_string.restype = ctypes.c_char_p
    lib.bsg_status_string.argtypes = [I]
    lib.bsg_quantize_mx.restype = I
    lib.bsg_quantize_mx.argtypes = [P, I64, I64, I64, I, I, I, P, P, P]
    lib.bsg_quantize_mx_bf16.restype = I
    lib.bsg_quantize_mx_bf16.argtypes = [P, I64, I64, I64, I, I, I, P, P, P]
    lib.bsg_gemm_amax.restype = I
    lib.bsg_gemm_amax.argtypes = [P, P, P, P, I, I, I, I64, I64, I64, I64, P, I, P,
                                  ctypes.POINTER(bsg_gemm_opts), P, SZ, P]
    lib.bsg_grouped_gemm_srelu.restype = I
    lib.bsg_grouped_gemm_srelu.argtypes = [P, P, P, P, I, I, I, I64, I64, I64, I64, P, P, P, F, P, P, I, P, P, I,
                                           P, P, P, ctypes.POINTER(bsg_gemm_opts), P, SZ, P]
    lib.bsg_grouped_discrete_workspace_size.restype = SZ
    lib.bsg_grouped_discrete_workspace_size.argtypes = [I64]
    lib.bsg_grouped_gemm_srelu_discrete.restype = I
    lib.bsg_grouped_gemm_srelu_discrete.argtypes = lib.bsg_grouped_gemm_srelu.argtypes
    lib.bsg_grouped_gemm_dswiglu.restype = I
    lib.bsg_grouped_gemm_dswiglu.argtypes = [P, P, P, P, I, I, I, I64, I64, I64, I64, P, P, P, P, P, I, P, P, P, I,
                                             P, P, P, P, ctypes.POINTER(bsg_gemm_opts), P, SZ, P]
    lib.bsg_rope_workspace_size.restype = SZ
    lib.bsg_rope_workspace_size.argtypes = [I64, I64, I64, I64]
    lib.bsg_gemm_rope_mxfp8.restype = I
    lib.bsg_gemm_rope_mxfp8.argtypes = [P, P, P, P, I, P, P, I64, I64, I64, I64, I64, P, P, P, P,
                                        ctypes.POINTER(bsg_gemm_opts), P, SZ, P]
    lib.bsg_gemm_rope_bf16.restype = I
    lib.bsg_gemm_rope_bf16.argtypes = [P, P, P, P, I64, I64, I64, I64, I64, P, P, P, P,
                                       ctypes.POINTER(bsg_gemm_opts), P, SZ, P]
    lib.bsg_selftest_wait_timeout.restype = I
    lib.bsg_selftest_wait_timeout.argtypes = [P, SZ, P]
    lib.bsg_gemm_amax_noalloc.restype = I
    lib.bsg_gemm_amax_noalloc.argtypes = [P, P, P, P, I, I, I, I64, I64, I64, I64, P, I, P,
                                          ctypes.POINTER(bsg_gemm_opts), P]
    lib.bsg_read_device_error.restype = I
    lib.bsg_read_device_error.argtypes = [P, P, U32P]
    lib.bsg_gemm_amax_noalloc_read_error.restype = I
    lib.bsg_gemm_amax_noalloc_read_error.argtypes = [P, U32P]
    return lib


_lib = _load()
LIBRARY_PATH = _lib._name


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _opts(tile_n=0, max_ctas=0, tanh_approx=False, validate_offsets=False, cta_pair=0, b_major="k"):
    o = bsg_gemm_opts()
    o.tile_n, o.max_ctas, o.tanh_approx, o.validate_offsets = tile_n, max_ctas, int(tanh_approx), int(validate_offsets)
    o.cta_pair = cta_pair
    o.b_major = {"k": 0, "n": 1}[b_major]
    return o


def _check(status, what):
    if status != OK:
        raise BsgError(status, what)


def bsg_workspace_size() -> int:
    return int(_lib.bsg_workspace_size())


def bsg_sf_bytes(batch: int, rows: int, k: int, sf_vec_size: int) -> int:
    return int(_lib.bsg_sf_bytes(batch, rows, k, sf_vec_size))


def bsg_status_string(status: int) -> str:
    return _lib.bsg_status_string(status).decode()


def bsg_quantize_mx(x, batch, rows, k, q_dtype, sf_vec_size, sf_dtype, q, sf, stream=None):
    _check(_lib.bsg_quantize_mx(_ptr(x), batch, rows, k, q_dtype, sf_vec_size, sf_dtype, _ptr(q), _ptr(sf),
                                _stream(stream)), "bsg_quantize_mx")


def bsg_quantize_mx_bf16(x, batch, rows, k, q_dtype, sf_vec_size, sf_dtype, q, sf, stream=None):
    _check(_lib.bsg_quantize_mx_bf16(_ptr(x), batch, rows, k, q_dtype, sf_vec_size, sf_dtype, _ptr(q), _ptr(sf),
                                     _stream(stream)), "bsg_quantize_mx_bf16")


def bsg_gemm_amax(a, b, sfa, sfb, ab_dtype, sf_dtype, sf_vec_size, m, n, k, l, c, c_dtype, amax, workspace,
                  workspace_bytes=None, stream=None, **opts):
    ws_bytes = bsg_workspace_size() if workspace_bytes is None else workspace_bytes
    o = _opts(**opts)
    _check(_lib.bsg_gemm_amax(_ptr(a), _ptr(b), _ptr(sfa), _ptr(sfb), ab_dtype, sf_dtype, sf_vec_size, m, n, k, l,
                              _ptr(c), c_dtype, _ptr(amax), ctypes.byref(o), _ptr(workspace), ws_bytes,
                              _stream(stream)), "bsg_gemm_amax")


def bsg_gemm_amax_noalloc(a, b, sfa, sfb, ab_dtype, sf_dtype, sf_vec_size, m, n, k, l, c, c_dtype, amax,
                          stream=None, **opts):
    """bsg_gemm_amax without a workspace argument: its scratch lives in a static device array
    of the library (for callers that cannot provide device memory; see include/bsg.h)."""
    o = _opts(**opts)
    _check(_lib.bsg_gemm_amax_noalloc(_ptr(a), _ptr(b), _ptr(sfa), _ptr(sfb), ab_dtype, sf_dtype, sf_vec_size, m, n,
                                      k, l, _ptr(c), c_dtype, _ptr(amax), ctypes.byref(o), _stream(stream)),
           "bsg_gemm_amax_noalloc")


def bsg_grouped_gemm_srelu(a, b, sfa, sfb, ab_dtype, sf_dtype, sf_vec_size, valid_m, n, k, num_experts,
                           padded_offsets, alpha, prob, tanh_clamp_scale, norm_const, c, c_dtype, d, d_col, d_dtype,
                           sfd_row, sfd_col, amax, workspace, workspace_bytes=None, stream=None, **opts):
    ws_bytes = bsg_workspace_size() if workspace_bytes is None else workspace_bytes
    o = _opts(**opts)
    s = 0.0 if tanh_clamp_scale is None else float(tanh_clamp_scale)
    _check(_lib.bsg_grouped_gemm_srelu(_ptr(a), _ptr(b), _ptr(sfa), _ptr(sfb), ab_dtype, sf_dtype, sf_vec_size,
                                       valid_m, n, k, num_experts, _ptr(padded_offsets), _ptr(alpha), _ptr(prob), s,
                                       _ptr(norm_const), _ptr(c), c_dtype, _ptr(d), _ptr(d_col), d_dtype,
                                       _ptr(sfd_row), _ptr(sfd_col), _ptr(amax), ctypes.byref(o), _ptr(workspace),
                                       ws_bytes, _stream(stream)), "bsg_grouped_gemm_srelu")


def bsg_grouped_discrete_workspace_size(num_experts: int) -> int:
    return int(_lib.bsg_grouped_discrete_workspace_size(num_experts))


def bsg_grouped_gemm_srelu_discrete(a, b_ptrs, sfa, sfb_ptrs, ab_dtype, sf_dtype, sf_vec_size, valid_m, n, k,
                                    num_experts, padded_offsets, alpha, prob, tanh_clamp_scale, norm_const, c, c_dtype,
                                    d, d_col, d_dtype, sfd_row, sfd_col, amax, workspace, workspace_bytes=None,
                                    stream=None, **opts):
    """b_ptrs / sfb_ptrs: device int64 arrays of the experts' B and SFB addresses."""
    ws_bytes = bsg_grouped_discrete_workspace_size(num_experts) if workspace_bytes is None else workspace_bytes
    o = _opts(**opts)
    s = 0.0 if tanh_clamp_scale is None else float(tanh_clamp_scale)
    _check(_lib.bsg_grouped_gemm_srelu_discrete(
        _ptr(a), _ptr(b_ptrs), _ptr(sfa), _ptr(sfb_ptrs), ab_dtype, sf_dtype, sf_vec_size, valid_m, n, k,
        num_experts, _ptr(padded_offsets), _ptr(alpha), _ptr(prob), s, _ptr(norm_const), _ptr(c), c_dtype, _ptr(d),
        _ptr(d_col), d_dtype, _ptr(sfd_row), _ptr(sfd_col), _ptr(amax), ctypes.byref(o), _ptr(workspace), ws_bytes,
        _stream(stream)), "bsg_grouped_gemm_srelu_discrete")


def bsg_grouped_gemm_dswiglu(a, b, sfa, sfb, ab_dtype, sf_dtype, sf_vec_size, valid_m, n, k, num_experts,
                             padded_offsets, alpha, beta, prob, c, c_dtype, norm_const, d_row, d_col, d_dtype,
                             sfd_row, sfd_col, dprob, amax, workspace, workspace_bytes=None, stream=None, **opts):
    ws_bytes = bsg_workspace_size() if workspace_bytes is None else workspace_bytes
    o = _opts(**opts)
    _check(_lib.bsg_grouped_gemm_dswiglu(
        _ptr(a), _ptr(b), _ptr(sfa), _ptr(sfb), ab_dtype, sf_dtype, sf_vec_size, valid_m, n, k, num_experts,
        _ptr(padded_offsets), _ptr(alpha), _ptr(beta), _ptr(prob), _ptr(c), c_dtype, _ptr(norm_const), _ptr(d_row),
        _ptr(d_col), d_dtype, _ptr(sfd_row), _ptr(sfd_col), _ptr(dprob), _ptr(amax), ctypes.byref(o),
        _ptr(workspace), ws_bytes, _stream(stream)), "bsg_grouped_gemm_dswiglu")


def bsg_rope_workspace_size(tokens: int, num_heads: int, head_dim: int, q_lora: int) -> int:
    return int(_lib.bsg_rope_workspace_size(tokens, num_heads, head_dim, q_lora))


def bsg_gemm_rope_mxfp8(x, x_scale, w, w_scale, scale_layout, cos, sin, tokens, q_lora, num_heads, head_dim, qk_rope,
                        out_fp8_row, out_scales_row, out_fp8_col, out_scales_col, workspace, workspace_bytes=None,
                        stream=None, **opts):
    ws_bytes = (bsg_rope_workspace_size(tokens, num_heads, head_dim, q_lora) if workspace_bytes is None
                else workspace_bytes)
    o = _opts(**opts)
    _check(_lib.bsg_gemm_rope_mxfp8(_ptr(x), _ptr(x_scale), _ptr(w), _ptr(w_scale), scale_layout, _ptr(cos), _ptr(sin),
                                    tokens, q_lora, num_heads, head_dim, qk_rope, _ptr(out_fp8_row),
                                    _ptr(out_scales_row), _ptr(out_fp8_col), _ptr(out_scales_col), ctypes.byref(o),
                                    _ptr(workspace), ws_bytes, _stream(stream)), "bsg_gemm_rope_mxfp8")


def bsg_gemm_rope_bf16(x, w, cos, sin, tokens, q_lora, num_heads, head_dim, qk_rope, out_fp8_row, out_scales_row,
                       out_fp8_col, out_scales_col, workspace, workspace_bytes=None, stream=None, **opts):
    ws_bytes = bsg_workspace_size() if workspace_bytes is None else workspace_bytes
    o = _opts(**opts)
    _check(_lib.bsg_gemm_rope_bf16(_ptr(x), _ptr(w), _ptr(cos), _ptr(sin), tokens, q_lora, num_heads, head_dim,
                                   qk_rope, _ptr(out_fp8_row), _ptr(out_scales_row), _ptr(out_fp8_col),
                                   _ptr(out_scales_col), ctypes.byref(o), _ptr(workspace), ws_bytes,
                                   _stream(stream)), "bsg_gemm_rope_bf16")


def bsg_selftest_wait_timeout(workspace, workspace_bytes=None, stream=None):
    """Runs the bounded-wait self-test (about two seconds); read the bits with bsg_read_device_error."""
    ws_bytes = bsg_workspace_size() if workspace_bytes is None else workspace_bytes
    _check(_lib.bsg_selftest_wait_timeout(_ptr(workspace), ws_bytes, _stream(stream)), "bsg_selftest_wait_timeout")


def bsg_read_device_error(workspace, stream=None) -> int:
    bits = ctypes.c_uint32(0)
    st = _lib.bsg_read_device_error(_ptr(workspace), _stream(stream), ctypes.byref(bits))
    if st not in (OK, 6):
        raise BsgError(st, "bsg_read_device_error")
    return int(bits.value)


def bsg_gemm_amax_noalloc_read_error(stream=None) -> int:
    """Error bits of the last bsg_gemm_amax_noalloc call on the current device (synchronises)."""
    bits = ctypes.c_uint32(0)
    st = _lib.bsg_gemm_amax_noalloc_read_error(_stream(stream), ctypes.byref(bits))
    if st not in (OK, 6):
        raise BsgError(st, "bsg_gemm_amax_noalloc_read_error")
    return int(bits.value)


def raw_status(fn_name: str, *args) -> int:
    """Calls an entry point with already-marshalled arguments and returns its status (tests of
    the host-side validation use this to see the code instead of an exception)."""
    return int(getattr(_lib, fn_name)(*args))

"""The C ABI library loads, exports every declared entry point, and validates arguments on the host.

These tests need no GPU: every rejected call returns its status before any CUDA call, and
the pointers passed are fake values that are never dereferenced.  A call that passes every
check would enqueue work on those fake pointers, so it runs only where no CUDA device is
present (it then stops at the device check).
"""
import ctypes
import os
import re

import pytest

import nvfp4_gemm_moe_gb300 as bsg
from nvfp4_gemm_moe_gb300 import build as bsg_build

OK, INVALID, UNSUPPORTED, ALIGN, ARCH, CUDA, DEVICE, BAD_OFFS, WORKSPACE = range(9)
P = 0x10000  # a fake, 16-byte aligned "device pointer" (never dereferenced by a rejected call)


def _no_device() -> bool:
    """True when no CUDA device is visible: only then may a call pass validation with fake pointers."""
    try:
        import torch
        return not torch.cuda.is_available()
    except ImportError:
        return True


def _declared_functions():
    src = open(bsg.HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:bsg_status|size_t|const char\s*\*)\s*(bsg_\w+)\s*\(", src, flags=re.M)))


def test_library_exports_every_declared_symbol():
    names = _declared_functions()
    assert {"bsg_quantize_mx", "bsg_gemm_amax", "bsg_grouped_gemm_srelu"} <= set(names)
    lib = ctypes.CDLL(bsg_build.build())
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"
    assert os.path.dirname(bsg.LIBRARY_PATH) == os.path.dirname(os.path.abspath(bsg.__file__))


def test_sizes_and_strings():
    assert bsg.bsg_workspace_size() == 256
    # (batch, ceil(rows/128), ceil(K/(4v)), 32, 4, 4)
    assert bsg.bsg_sf_bytes(1, 256, 256, 32) == 1 * 2 * 2 * 512
    assert bsg.bsg_sf_bytes(4, 8192, 8192, 32) == 4 * 64 * 64 * 512
    assert bsg.bsg_sf_bytes(1, 130, 96, 16) == 2 * 2 * 512
    assert bsg.bsg_sf_bytes(0, 1, 1, 32) == 0
    assert bsg.bsg_status_string(0) == "BSG_OK"
    assert bsg.bsg_status_string(7) == "BSG_ERR_BAD_OFFSETS"


def _quant(name="bsg_quantize_mx", **kw):
    a = dict(x=P, batch=1, rows=128, k=256, q=0x1, v=32, sf=0, qp=P, sfp=P, stream=None)
    a.update(kw)
    return bsg.raw_status(name, a["x"], a["batch"], a["rows"], a["k"], a["q"], a["v"], a["sf"],
                          a["qp"], a["sfp"], a["stream"])


def test_quantize_bf16_validation():
    """The bf16-input entry shares the fp32 entry's checks."""
    E4M3, E2M1 = bsg.E4M3, bsg.E2M1

    def q(**kw):
        a = dict(q=E4M3, v=32, sf=bsg.SF_UE8M0)
        a.update(kw)
        return _quant("bsg_quantize_mx_bf16", **a)
    assert q(x=None) == INVALID
    assert q(v=16) == INVALID                         # FP8 needs v = 32
    assert q(q=bsg.E5M2) == UNSUPPORTED
    assert q(k=48) == INVALID
    assert q(x=P + 8) == ALIGN
    assert q(q=E2M1, v=16, sf=bsg.SF_UE4M3, k=48) == ALIGN
    if _no_device():
        assert q() in (ARCH, CUDA)
        assert q(q=E2M1, v=16, sf=bsg.SF_UE4M3) in (ARCH, CUDA)


def test_quantize_validation():
    E4M3, E2M1, E5M2 = bsg.E4M3, bsg.E2M1, bsg.E5M2
    assert _quant(q=E4M3, v=32, sf=bsg.SF_UE8M0, x=None) == INVALID
    assert _quant(q=E4M3, v=16, sf=bsg.SF_UE8M0) == INVALID         # FP8 needs v = 32
    assert _quant(q=E2M1, v=32, sf=bsg.SF_UE4M3) == INVALID         # E4M3 scales need v = 16
    assert _quant(q=E5M2, v=32, sf=bsg.SF_UE8M0) == UNSUPPORTED
    assert _quant(q=E2M1, v=32, sf=bsg.SF_UE8M0) == UNSUPPORTED     # MXFP4
    assert _quant(q=E4M3, v=32, sf=bsg.SF_UE8M0, k=48) == INVALID   # K not a whole number of blocks
    assert _quant(q=E2M1, v=16, sf=bsg.SF_UE4M3, k=48) == ALIGN     # K/2 bytes not a multiple of 16
    assert _quant(q=E4M3, v=32, sf=bsg.SF_UE8M0, x=P + 4) == ALIGN
    assert _quant(q=E4M3, v=32, sf=bsg.SF_UE8M0, rows=0) == INVALID


def _opts():
    return ctypes.byref(bsg.bsg_gemm_opts())


def _dense(**kw):
    a = dict(a=P, b=P, sfa=P, sfb=P, ab=bsg.E4M3, sf=bsg.SF_UE8M0, v=32, m=256, n=256, k=256, l=1, c=P,
             ck=bsg.BF16, amax=P, ws=P, wsb=256)
    a.update(kw)
    return bsg.raw_status("bsg_gemm_amax", a["a"], a["b"], a["sfa"], a["sfb"], a["ab"], a["sf"], a["v"], a["m"],
                          a["n"], a["k"], a["l"], a["c"], a["ck"], a["amax"], _opts(), a["ws"], a["wsb"], None)


def test_dense_validation():
    assert _dense(a=None) == INVALID
    assert _dense(amax=None) == INVALID
    assert _dense(ws=None) == WORKSPACE
    assert _dense(wsb=128) == WORKSPACE
    assert _dense(m=0) == INVALID
    assert _dense(k=48) == INVALID
    assert _dense(k=16 * 33) == INVALID                # not a multiple of 32
    assert _dense(ck=bsg.E5M2) == UNSUPPORTED
    assert _dense(ck=bsg.E4M3) == UNSUPPORTED         # FP8 C with FP8 operands is disabled
    assert _dense(ck=bsg.E2M1) == UNSUPPORTED         # FP4 C needs FP4 operands
    assert _dense(ck=bsg.F16, n=4) == ALIGN           # 8 bytes per row of C
    assert _dense(ab=bsg.E2M1, sf=bsg.SF_UE4M3, v=16, ck=bsg.E2M1, n=16) == ALIGN  # 8 bytes per row
    assert _dense(n=4) == ALIGN                         # 4 bf16 = 8 bytes per row of C
    assert _dense(c=P + 8) == ALIGN
    assert _dense(ws=P + 16) == ALIGN                   # workspace is 256-byte aligned
    assert _dense(ab=bsg.E2M1, sf=bsg.SF_UE4M3, v=16, k=48) == ALIGN  # 24-byte rows
    assert _dense(m=1 << 31) == INVALID
    # a valid call on a machine without a usable sm_103 device stops at the device check
    if _no_device():
        st = _dense()
        assert st in (OK, ARCH, CUDA)


def _grouped(**kw):
    a = dict(a=P, b=P, sfa=P, sfb=P, ab=bsg.E4M3, sf=bsg.SF_UE8M0, v=32, vm=512, n=256, k=256, L=2, offs=P,
             alpha=P, prob=P, s=0.0, nc=None, c=P, ck=bsg.BF16, d=P, dcol=None, dk=bsg.BF16, sfr=None, sfc=None,
             amax=P, ws=P, wsb=256)
    a.update(kw)
    return bsg.raw_status("bsg_grouped_gemm_srelu", a["a"], a["b"], a["sfa"], a["sfb"], a["ab"], a["sf"], a["v"],
                          a["vm"], a["n"], a["k"], a["L"], a["offs"], a["alpha"], a["prob"], ctypes.c_float(a["s"]),
                          a["nc"], a["c"], a["ck"], a["d"], a["dcol"], a["dk"], a["sfr"], a["sfc"], a["amax"],
                          _opts(), a["ws"], a["wsb"], None)


def test_grouped_validation():
    assert _grouped(prob=None) == INVALID                # prob is required
    assert _grouped(vm=300) == INVALID                   # valid_m must be a multiple of 256
    assert _grouped(L=0) == INVALID and _grouped(L=1025) == INVALID
    assert _grouped(amax=None) == INVALID                # bf16 D needs the per-expert amax
    assert _grouped(dcol=P) == INVALID                   # D_col only with E4M3 D
    assert _grouped(dk=bsg.E4M3) == INVALID              # E4M3 D needs d_col, SFD and norm_const
    assert _grouped(dk=bsg.E4M3, dcol=P, sfr=P, sfc=P, nc=P, amax=None, n=48) == INVALID  # n % 32
    assert _grouped(dk=bsg.E5M2) == UNSUPPORTED
    assert _grouped(ck=bsg.E4M3) == UNSUPPORTED
    assert _grouped(dk=bsg.F32, n=2) == ALIGN             # 8 bytes per row of D
    assert _grouped(dk=bsg.E4M3, dcol=P, sfr=P, sfc=P, nc=P, amax=None, ab=bsg.E2M1, sf=bsg.SF_UE4M3,
                    v=16) == UNSUPPORTED                  # E4M3 D only with E4M3 operands
    assert _grouped(s=float("nan")) == INVALID
    assert _grouped(ws=None) == WORKSPACE
    assert _grouped(offs=P + 2) == ALIGN
    if _no_device():
        st = _grouped()
        assert st in (OK, ARCH, CUDA)


def _discrete(**kw):
    a = dict(a=P, bp=P, sfa=P, sp=P, L=2, ws=P, wsb=256 + 2 * 128, d=P)
    a.update(kw)
    return bsg.raw_status("bsg_grouped_gemm_srelu_discrete", a["a"], a["bp"], a["sfa"], a["sp"], bsg.E4M3,
                          bsg.SF_UE8M0, 32, 512, 256, 256, a["L"], P, P, P, ctypes.c_float(0.0), None, P, bsg.BF16,
                          a["d"], None, bsg.BF16, None, None, P, _opts(), a["ws"], a["wsb"], None)


def test_discrete_validation():
    # the error word plus one 128-byte TMA descriptor per expert
    assert bsg.bsg_grouped_discrete_workspace_size(1) == 256 + 128
    assert bsg.bsg_grouped_discrete_workspace_size(32) == 256 + 32 * 128
    assert _discrete(bp=None) == INVALID
    assert _discrete(sp=None) == INVALID
    assert _discrete(wsb=256) == WORKSPACE                # too small for the descriptors
    assert _discrete(bp=P + 4) == ALIGN                    # int64 array
    assert _discrete(ws=P + 64) == ALIGN
    assert _discrete(L=0) == INVALID
    if _no_device():
        st = _discrete()
        assert st in (OK, ARCH, CUDA)


def _dsw(**kw):
    a = dict(a=P, b=P, sfa=P, sfb=P, ab=bsg.E4M3, sf=bsg.SF_UE8M0, v=32, vm=512, n=256, k=256, L=2, offs=P,
             alpha=P, beta=P, prob=P, c=P, ck=bsg.BF16, nc=None, d=P, dcol=None, dk=bsg.BF16, sfr=None, sfc=None,
             dprob=P, amax=P, ws=P, wsb=256)
    a.update(kw)
    return bsg.raw_status("bsg_grouped_gemm_dswiglu", a["a"], a["b"], a["sfa"], a["sfb"], a["ab"], a["sf"], a["v"],
                          a["vm"], a["n"], a["k"], a["L"], a["offs"], a["alpha"], a["beta"], a["prob"], a["c"],
                          a["ck"], a["nc"], a["d"], a["dcol"], a["dk"], a["sfr"], a["sfc"], a["dprob"], a["amax"],
                          _opts(), a["ws"], a["wsb"], None)


def test_dswiglu_validation():
    assert _dsw(c=None) == INVALID                       # the forward intermediate is an input
    assert _dsw(beta=None) == INVALID and _dsw(dprob=None) == INVALID
    assert _dsw(n=48) == INVALID                         # 32-column input / gate blocks
    assert _dsw(L=513) == INVALID                        # 2 * L amax values in shared memory
    assert _dsw(amax=None) == INVALID                    # float D needs the (L, 2) amax
    assert _dsw(dk=bsg.E4M3) == INVALID                  # E4M3 D needs d_col, SFD and norm_const
    assert _dsw(dk=bsg.E4M3, dcol=P, sfr=P, sfc=P, nc=P, ab=bsg.E2M1, sf=bsg.SF_UE4M3, v=16) == UNSUPPORTED
    assert _dsw(ck=bsg.E2M1) == UNSUPPORTED
    assert _dsw(dk=bsg.E5M2) == UNSUPPORTED
    assert _dsw(dprob=P + 2) == ALIGN
    assert _dsw(c=P + 8) == ALIGN
    assert _dsw(wsb=16) == WORKSPACE
    if _no_device():
        st = _dsw()
        assert st in (OK, ARCH, CUDA)
        st = _dsw(dk=bsg.E4M3, dcol=P, sfr=P, sfc=P, nc=P, amax=None, ck=bsg.E4M3)
        assert st in (OK, ARCH, CUDA)


def _rope(name="bsg_gemm_rope_mxfp8", cta_pair=0, tile_n=0, **kw):
    a = dict(x=P, w=P, cos=P, sin=P, tokens=256, q=256, h=2, hd=192, r=64, orow=P, srow=P, ocol=P, scol=P,
             layout=0, ws=P, wsb=256)
    a.update(kw)
    o = bsg._opts(cta_pair=cta_pair, tile_n=tile_n)
    tail = (a["tokens"], a["q"], a["h"], a["hd"], a["r"], a["orow"], a["srow"], a["ocol"], a["scol"], ctypes.byref(o),
            a["ws"], a["wsb"], None)
    if name == "bsg_gemm_rope_bf16":
        return bsg.raw_status(name, a["x"], a["w"], a["cos"], a["sin"], *tail)
    return bsg.raw_status(name, a["x"], P, a["w"], P, a["layout"], a["cos"], a["sin"], *tail)


def test_rope_validation():
    for name in ("bsg_gemm_rope_mxfp8", "bsg_gemm_rope_bf16"):
        assert _rope(name, x=None) == INVALID and _rope(name, scol=None) == INVALID
        assert _rope(name, tokens=200) == INVALID and _rope(name, tokens=0) == INVALID
        assert _rope(name, hd=128) == UNSUPPORTED and _rope(name, r=32) == UNSUPPORTED
        assert _rope(name, wsb=128) == WORKSPACE and _rope(name, ws=None) == WORKSPACE
        assert _rope(name, orow=P + 8) == ALIGN and _rope(name, cos=P + 2) == ALIGN
        assert _rope(name, ws=P + 16) == ALIGN
    assert _rope(q=48) == INVALID                     # MXFP8: whole 32-value scale blocks
    assert _rope(layout=2) == INVALID
    assert _rope(layout=1) == WORKSPACE               # the plain scales are repacked in the workspace
    assert _rope(cta_pair=2, tokens=128) == INVALID   # pairs need tokens and heads * 192 in 256s
    assert _rope(cta_pair=2, h=3) == INVALID          # 256-wide pair tiles: heads * 192 % 256 != 0
    bf = "bsg_gemm_rope_bf16"
    assert _rope(bf, q=12) == INVALID                 # bf16 rows must be 16-byte multiples
    assert _rope(bf, q=4) == INVALID
    assert _rope(bf, cta_pair=2, tokens=128) == INVALID  # pair tiles need tokens % 256 == 0
    if _no_device():
        assert _rope() in (OK, ARCH, CUDA)
        assert _rope(bf, q=72) in (OK, ARCH, CUDA)
        assert _rope(cta_pair=2, h=3, tile_n=192) in (OK, ARCH, CUDA)  # 256 x 192 pair tiles
        assert _rope(bf, cta_pair=2) in (OK, ARCH, CUDA)


def test_selftest_validation():
    assert bsg.raw_status("bsg_selftest_wait_timeout", None, 256, None) == WORKSPACE
    assert bsg.raw_status("bsg_selftest_wait_timeout", P, 16, None) == WORKSPACE
    assert bsg.raw_status("bsg_selftest_wait_timeout", P + 16, 256, None) == ALIGN
    if _no_device():
        assert bsg.raw_status("bsg_selftest_wait_timeout", P, 256, None) in (ARCH, CUDA)


def test_noalloc_validation():
    def call(**kw):
        a = dict(a=P, c=P, amax=P, n=256)
        a.update(kw)
        return bsg.raw_status("bsg_gemm_amax_noalloc", a["a"], P, P, P, bsg.E4M3, bsg.SF_UE8M0, 32, 256, a["n"],
                              256, 1, a["c"], bsg.BF16, a["amax"], _opts(), None)
    assert call(a=None) in (INVALID, CUDA)
    assert call(n=4) in (ALIGN, CUDA)
    # the GEMM's scratch fits the library's static array (also a compile-time check in the library)
    assert bsg.bsg_workspace_size() <= 256
    assert "#define BSG_NOALLOC_SCRATCH_BYTES 256" in open(bsg.HEADER).read()
    assert bsg.raw_status("bsg_gemm_amax_noalloc_read_error", None, None) == INVALID
    if _no_device():
        import ctypes as ct
        bits = ct.c_uint32(7)
        assert bsg.raw_status("bsg_gemm_amax_noalloc_read_error", None, ct.byref(bits)) == CUDA


def test_binding_raises_on_bad_status():
    with pytest.raises(bsg.BsgError) as ei:
        bsg.bsg_quantize_mx(P, 1, 128, 48, bsg.E4M3, 32, bsg.SF_UE8M0, P, P, stream=0)
    assert ei.value.status == INVALID

"""Float64 CPU oracle for the block-scaled GEMM hot path -- TEST INFRASTRUCTURE.

Plain, slow, obviously-correct restatements of what the pages define:

* ``formats``   -- E4M3 / E2M1 / E8M0 / UE4M3 codecs (decode by formula, encode by
                   round-to-nearest-even decided on exact values);
* ``sf_layout`` -- the 128x4 scale-factor atom layout and its physical byte order;
* ``quantize``  -- the MXFP8 / NVFP4 input quantiser of the workloads and the
                   per-block dequantisation;
* ``gemm``      -- dense batched GEMM + global amax, grouped GEMM + prob-gated
                   sReLU (optional tanh clamp), per-expert amax and the row/column
                   MXFP8 re-quantisation of D;
* ``dswiglu``   -- grouped GEMM + dSwiGLU backward epilogue (32-column
                   input/gate interleave, dprob, (L, 2) amax, FP8 D);
* ``rope``      -- dense MXFP8 projection GEMM + per-head interleaved-in / halves-out
                   RoPE + dual-direction MXFP8 with plain scale layouts.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  It shares no
code with the CUDA library and never imports it.

Pinning status: every function is pinned by a ``-m "not gpu"`` test against
something other than itself (library decoders, closed forms, brute force,
invariants; the dSwiGLU epilogue against torch autograd through torch's SiLU, the
RoPE rotation against complex multiplication); see ``tests/test_oracle_*.py``.  One reading remains unpinned
against the pages' own implementation because the pages print no outputs: the
row order inside a 128-row scale-factor atom (``sf_layout``), "parity unpinned"
in that sense only.
"""
from . import formats, sf_layout, quantize, gemm, dswiglu, rope  # noqa: F401

"""Seeded synthetic inputs for the block-scaled GEMM workloads.

This module holds random draws and workload recipes only: shapes, value
distributions, expert routing counts and the 256-row padding of each expert's
row range.  It contains none of the method's arithmetic (no quantisation, no
scale-factor layout, no GEMM, no epilogue); the float64 oracle and the CUDA
library each derive everything else from the fp32 tensors produced here.

Every value is a pure function of ``(seed, stream, flat index)``: the flat range
of a tensor is cut into chunks of ``CHUNK`` elements and chunk ``c`` is drawn by
its own PCG64 generator seeded with ``SeedSequence([seed, stream, c])``.  So a
few rows of a multi-gigabyte operand can be regenerated alone (for sampled
parity checks) and the full tensor can be filled by several threads with the
same result.

The five workloads follow the shapes named by the pages' dense GEMM + Amax and
grouped GEMM + sReLU operations (both "Shapes" sections); the recipes
(distributions, routing, padding) are the ones stated for each workload below.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import math
import os

import numpy as np

CHUNK = 1 << 20

# stream ids: one per tensor kind so tensors never share random numbers
S_A, S_B, S_ALPHA, S_PROB, S_ROUTE, S_C, S_BETA = 1, 2, 3, 4, 5, 6, 7
SEQ_LEN_ROPE = 4096  # positions of the RoPE workload restart every 4096 tokens (one sequence)

PAD = 256  # expert row ranges are padded to multiples of 256 rows


def _chunk_rng(seed: int, stream: int, chunk: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, chunk])))


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def normal_f32(seed: int, stream: int, start: int, stop: int) -> np.ndarray:
    """Standard normal float32 values for flat indices ``[start, stop)``."""
    n = stop - start
    out = np.empty(n, dtype=np.float32)
    if n <= 0:
        return out
    c0, c1 = start // CHUNK, (stop - 1) // CHUNK

    def fill(c: int) -> None:
        lo, hi = c * CHUNK, (c + 1) * CHUNK
        buf = _chunk_rng(seed, stream, c).standard_normal(CHUNK, dtype=np.float32)
        a, b = max(lo, start), min(hi, stop)
        out[a - start:b - start] = buf[a - lo:b - lo]

    chunks = range(c0, c1 + 1)
    if len(chunks) == 1:
        fill(c0)
    else:
        with _cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, chunks))
    return out


def normal_f32_rows(seed: int, stream: int, rows, row_len: int) -> np.ndarray:
    """Rows ``rows`` (flat row indices) of a row-major normal tensor with ``row_len`` columns.

    Same values as slicing ``normal_f32`` over the whole tensor; every chunk the rows touch
    is drawn once.
    """
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    out = np.empty((rows.size, row_len), dtype=np.float32)
    if rows.size == 0 or row_len == 0:
        return out
    starts = rows * row_len
    chunks = sorted({int(c) for s in starts for c in range(s // CHUNK, (s + row_len - 1) // CHUNK + 1)})

    def draw(c: int) -> np.ndarray:
        return _chunk_rng(seed, stream, c).standard_normal(CHUNK, dtype=np.float32)

    if len(chunks) == 1:
        bufs = {chunks[0]: draw(chunks[0])}
    else:
        with _cf.ThreadPoolExecutor(_threads()) as ex:
            bufs = dict(zip(chunks, ex.map(draw, chunks)))
    for i, s in enumerate(starts):
        pos = 0
        while pos < row_len:
            c, off = divmod(int(s) + pos, CHUNK)
            take = min(row_len - pos, CHUNK - off)
            out[i, pos:pos + take] = bufs[c][off:off + take]
            pos += take
    return out


def uniform_f32(seed: int, stream: int, n: int, lo: float, hi: float) -> np.ndarray:
    """``n`` float32 values uniform in [lo, hi) (one generator; n is small)."""
    u = _chunk_rng(seed, stream, 0).random(n, dtype=np.float32)
    return (np.float32(lo) + np.float32(hi - lo) * u).astype(np.float32)


# ----------------------------------------------------------------------------
# dense workloads


@dataclasses.dataclass(frozen=True)
class Dense:
    """Batched dense block-scaled GEMM + amax workload: A (L,M,K), B (L,N,K)."""
    name: str
    m: int
    n: int
    k: int
    l: int
    fmt: str            # "mxfp8" (E4M3 codes, E8M0 scales, v=32) or "nvfp4" (E2M1, UE4M3, v=16)
    c_dtype: str        # "f32" or "bf16"
    boost_every: int = 0  # if >0: K-blocks kb with kb % boost_every == boost_every-1 of A are x2^6
    seed: int = 0

    @property
    def sf_vec(self) -> int:
        return 32 if self.fmt == "mxfp8" else 16

    @property
    def flops(self) -> float:
        return 2.0 * self.m * self.n * self.k * self.l

    def a_rows(self, rows: np.ndarray | None = None) -> np.ndarray:
        """fp32 A as (L, M, K); with ``rows`` (flat indices l*M+m) only those rows."""
        return self._rows(S_A, self.m, rows, boost=True)

    def b_rows(self, rows: np.ndarray | None = None) -> np.ndarray:
        return self._rows(S_B, self.n, rows, boost=False)

    def _rows(self, stream, nrows, rows, boost):
        k = self.k
        if rows is None:
            x = normal_f32(self.seed, stream, 0, self.l * nrows * k).reshape(self.l, nrows, k)
        else:
            x = normal_f32_rows(self.seed, stream, rows, k)
        if boost and self.boost_every:
            v, e = self.sf_vec, self.boost_every
            kb = np.arange(k) // v
            x[..., (kb % e) == e - 1] *= np.float32(64.0)
        return x


# ----------------------------------------------------------------------------
# grouped (MoE) workloads


@dataclasses.dataclass(frozen=True)
class Grouped:
    """Grouped block-scaled GEMM + sReLU workload over 256-padded expert row ranges."""
    name: str
    experts: int
    k: int
    n: int
    routed_rows: int
    skew: str              # "uniform" or "zipf1.2"
    d_dtype: str           # "bf16" or "e4m3"
    tanh_clamp: float | None = None
    seed: int = 0
    fmt: str = "mxfp8"

    @property
    def sf_vec(self) -> int:
        return 32 if self.fmt == "mxfp8" else 16

    def counts(self) -> np.ndarray:
        """Routed rows per expert: one seeded multinomial draw."""
        g = np.arange(self.experts, dtype=np.float64)
        if self.skew == "uniform":
            p = np.full(self.experts, 1.0 / self.experts)
        elif self.skew.startswith("zipf"):
            s = float(self.skew[4:])
            w = (g + 1.0) ** (-s)
            p = w / w.sum()
        elif self.skew.startswith("fixed:"):
            return np.array([int(c) for c in self.skew[6:].split(",")], dtype=np.int64)
        else:
            raise ValueError(self.skew)
        rng = _chunk_rng(self.seed, S_ROUTE, 0)
        return rng.multinomial(self.routed_rows, p).astype(np.int64)

    def padded_offsets(self) -> np.ndarray:
        """int32 cumulative ends of each expert's range, each padded up to 256 rows."""
        c = self.counts()
        padded = (c + PAD - 1) // PAD * PAD
        return np.cumsum(padded).astype(np.int32)

    @property
    def valid_m(self) -> int:
        return int(self.padded_offsets()[-1])

    @property
    def flops(self) -> float:
        return 2.0 * self.valid_m * self.n * self.k

    def routed_mask(self) -> np.ndarray:
        """Boolean (valid_m,): True for routed rows, False for padding rows."""
        c = self.counts()
        ends = self.padded_offsets().astype(np.int64)
        mask = np.zeros(int(ends[-1]), dtype=bool)
        begin = 0
        for g in range(self.experts):
            mask[begin:begin + c[g]] = True
            begin = int(ends[g])
        return mask

    def a_rows(self, rows: np.ndarray | None = None) -> np.ndarray:
        """fp32 A (valid_m, K): N(0,1)/sqrt(K) on routed rows, zero on padding rows."""
        k, vm = self.k, self.valid_m
        scale = np.float32(1.0 / math.sqrt(k))
        mask = self.routed_mask()
        if rows is None:
            x = normal_f32(self.seed, S_A, 0, vm * k).reshape(vm, k)
            x *= scale
            x[~mask] = 0.0
        else:
            x = normal_f32_rows(self.seed, S_A, rows, k)
            x *= scale
            x[~mask[np.asarray(rows)]] = 0.0
        return x

    def b_rows(self, rows: np.ndarray | None = None) -> np.ndarray:
        """fp32 B (L, N, K) as N(0,1)/sqrt(K); with ``rows`` (flat g*N+n) only those rows."""
        k = self.k
        scale = np.float32(1.0 / math.sqrt(k))
        if rows is None:
            x = normal_f32(self.seed, S_B, 0, self.experts * self.n * k).reshape(self.experts, self.n, k)
        else:
            x = normal_f32_rows(self.seed, S_B, rows, k)
        x *= scale
        return x

    def alpha(self) -> np.ndarray:
        return uniform_f32(self.seed, S_ALPHA, self.experts, 0.5, 2.0)

    def prob(self) -> np.ndarray:
        return uniform_f32(self.seed, S_PROB, self.valid_m, 0.0, 1.0)


@dataclasses.dataclass(frozen=True)
class GroupedDswiglu(Grouped):
    """Grouped GEMM + dSwiGLU backward workload: the grouped operands plus the stored forward
    intermediate C (valid_m, 2N) and the per-expert scale beta of C."""
    c_dtype: str = "bf16"   # element type C is stored in

    def c_rows(self, rows: np.ndarray | None = None) -> np.ndarray:
        """fp32 C (valid_m, 2N) as 3 N(0,1) on routed rows (gates reach the sigmoid's tails),
        zero on padding rows (the forward pass left them zero)."""
        two_n, vm = 2 * self.n, self.valid_m
        mask = self.routed_mask()
        if rows is None:
            x = normal_f32(self.seed, S_C, 0, vm * two_n).reshape(vm, two_n)
            x *= np.float32(3.0)
            x[~mask] = 0.0
        else:
            x = normal_f32_rows(self.seed, S_C, rows, two_n)
            x *= np.float32(3.0)
            x[~mask[np.asarray(rows)]] = 0.0
        return x

    def beta(self) -> np.ndarray:
        return uniform_f32(self.seed, S_BETA, self.experts, 0.5, 2.0)


@dataclasses.dataclass(frozen=True)
class RopeProj:
    """Dense projection + per-head RoPE + dual-direction MXFP8 workload: x (tokens, q_lora),
    w (heads * head_dim, q_lora) ([out, in]), rotary tables (tokens, qk_rope).  fmt "mxfp8": the
    operands are quantised to MXFP8; fmt "bf16": they are the fp32 draws rounded to bf16."""
    name: str
    tokens: int
    q_lora: int
    heads: int
    head_dim: int
    qk_rope: int
    seed: int = 0
    fmt: str = "mxfp8"

    @property
    def n(self) -> int:
        return self.heads * self.head_dim

    @property
    def flops(self) -> float:
        return 2.0 * self.tokens * self.q_lora * self.n

    def x_rows(self, rows: np.ndarray | None = None) -> np.ndarray:
        """fp32 x (tokens, q_lora) as N(0,1)."""
        if rows is None:
            return normal_f32(self.seed, S_A, 0, self.tokens * self.q_lora).reshape(self.tokens, self.q_lora)
        return normal_f32_rows(self.seed, S_A, rows, self.q_lora)

    def w_rows(self, rows: np.ndarray | None = None) -> np.ndarray:
        """fp32 w (heads * head_dim, q_lora) as N(0,1)/sqrt(q_lora)."""
        scale = np.float32(1.0 / math.sqrt(self.q_lora))
        if rows is None:
            x = normal_f32(self.seed, S_B, 0, self.n * self.q_lora).reshape(self.n, self.q_lora)
        else:
            x = normal_f32_rows(self.seed, S_B, rows, self.q_lora)
        x *= scale
        return x

    def tables(self) -> tuple[np.ndarray, np.ndarray]:
        """fp32 cos, sin (tokens, qk_rope): angle position * 10000^(-2j/qk_rope) for pair j, the
        same angle in both halves; positions restart every SEQ_LEN_ROPE tokens."""
        half = self.qk_rope // 2
        pos = (np.arange(self.tokens) % SEQ_LEN_ROPE).astype(np.float64)
        inv_freq = 10000.0 ** (-2.0 * np.arange(half) / self.qk_rope)
        ang = pos[:, None] * inv_freq[None, :]
        ang = np.concatenate([ang, ang], axis=1)
        return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


# The five named workloads.  The first is small enough for the oracle to finish
# in seconds; the second is the large batched dense one throughput is quoted on.
DENSE_MXFP8_256 = Dense("dense_mxfp8_m256_n256_k256_l1", 256, 256, 256, 1, "mxfp8", "f32")
DENSE_MXFP8_8192 = Dense("dense_mxfp8_m8192_n8192_k8192_l4", 8192, 8192, 8192, 4, "mxfp8", "bf16",
                         boost_every=7)
# one batch of the large dense workload (same draws as its batch 0): the case profiled under ncu
DENSE_MXFP8_8192_L1 = dataclasses.replace(DENSE_MXFP8_8192, name="dense_mxfp8_m8192_n8192_k8192_l1", l=1)
DENSE_NVFP4_16384 = Dense("dense_nvfp4_m16384_n16384_k8192_l1", 16384, 16384, 8192, 1, "nvfp4", "bf16")
GROUPED_SRELU_E32 = Grouped("grouped_mxfp8_srelu_e32_k7168_n2048", 32, 7168, 2048, 32768, "uniform", "bf16")
GROUPED_SRELU_E32_CLAMP = dataclasses.replace(GROUPED_SRELU_E32, name=GROUPED_SRELU_E32.name + "_tanh32",
                                              tanh_clamp=32.0)
GROUPED_FP8D_E128 = Grouped("grouped_mxfp8_fp8d_e128_k4096_n4096", 128, 4096, 4096, 65536, "zipf1.2", "e4m3")

# the E4M3-D kernel on 32 experts (same K, N, routing skew): the case its ncu capture runs on,
# a few GB on the device instead of the 128-expert workload's twelve
GROUPED_FP8D_E32 = Grouped("grouped_mxfp8_fp8d_e32_k4096_n4096", 32, 4096, 4096, 16384, "zipf1.2", "e4m3")
# the backward of the E32 expert layer: dSwiGLU over the same routing, ref N = 2048 (C and D 4096 wide)
GROUPED_DSWIGLU_E32 = GroupedDswiglu("grouped_mxfp8_dswiglu_e32_k7168_n2048", 32, 7168, 2048, 32768, "uniform",
                                     "bf16")
GROUPED_DSWIGLU_E32_FP8D = dataclasses.replace(GROUPED_DSWIGLU_E32, name="grouped_mxfp8_dswiglu_fp8d_e32_k7168_n2048",
                                               d_dtype="e4m3")

# the DeepSeek-V3 MLA Q up-projection: 128 heads of 128 + 64 features from a 1536-wide latent
ROPE_PROJ_T16384 = RopeProj("rope_proj_mxfp8_t16384_q1536_h128_d192", 16384, 1536, 128, 192, 64)
# the same projection with bf16 operands
ROPE_PROJ_BF16_T16384 = RopeProj("rope_proj_bf16_t16384_q1536_h128_d192", 16384, 1536, 128, 192, 64, fmt="bf16")

ALL = {w.name: w for w in (DENSE_MXFP8_256, DENSE_MXFP8_8192, DENSE_MXFP8_8192_L1, DENSE_NVFP4_16384, GROUPED_SRELU_E32,
                           GROUPED_SRELU_E32_CLAMP, GROUPED_FP8D_E128, GROUPED_FP8D_E32, GROUPED_DSWIGLU_E32,
                           GROUPED_DSWIGLU_E32_FP8D, ROPE_PROJ_T16384, ROPE_PROJ_BF16_T16384)}

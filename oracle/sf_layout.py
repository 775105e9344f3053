"""Scale-factor atom layout (oracle; test infrastructure).

"GEMM + Amax (SM100)", Shapes: SFA has the logical shape
(32, 4, ceil(M/128), 4, ceil(K/(4*v)), L); "Using JAX arrays": it is the
C-contiguous physical allocation (L, ceil(M/128), ceil(K/(4*v)), 32, 4, 4)
permuted by (3, 4, 1, 5, 2, 0).  "Grouped GEMM + sReLU (SM100)", Shapes, uses the
same layout for SFA/SFB/SFD_row/SFD_col with (rows, blocks) = (valid_m, K/v),
(N, K/v), (valid_m, N/32) and (N, valid_m/32).

Reading taken where the pages are silent: a logical index (i0, i1, mt, k0, kt, l)
names row ``mt*128 + i1*32 + i0`` and scale block ``kt*4 + k0`` (first mode
fastest within each nested mode).  Hence the byte of (row r, block kb, batch l) is

    ((((l*MT + r//128)*KT + kb//4)*32 + r%32)*4 + (r%128)//32)*4 + kb%4.

Bytes of the padded extent (rows >= rows, blocks >= blocks) are zero.
"""
from __future__ import annotations

import numpy as np


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def physical_shape(rows: int, blocks: int, batch: int = 1) -> tuple:
    return (batch, ceil_div(rows, 128), ceil_div(blocks, 4), 32, 4, 4)


def nbytes(rows: int, blocks: int, batch: int = 1) -> int:
    return int(np.prod(physical_shape(rows, blocks, batch)))


def offset(r, kb, l, rows: int, blocks: int):
    """Byte offset of (row r, scale block kb, batch l) in the physical buffer."""
    mt_n, kt_n = ceil_div(rows, 128), ceil_div(blocks, 4)
    r = np.asarray(r, dtype=np.int64)
    kb = np.asarray(kb, dtype=np.int64)
    l = np.asarray(l, dtype=np.int64)
    return (((((l * mt_n + r // 128) * kt_n + kb // 4) * 32 + r % 32) * 4 + (r % 128) // 32) * 4 + kb % 4)


def pack(sf: np.ndarray) -> np.ndarray:
    """Logical per-block scale bytes (batch, rows, blocks) -> flat physical uint8 buffer."""
    sf = np.asarray(sf, dtype=np.uint8)
    batch, rows, blocks = sf.shape
    out = np.zeros(nbytes(rows, blocks, batch), dtype=np.uint8)
    l, r, kb = np.meshgrid(np.arange(batch), np.arange(rows), np.arange(blocks), indexing="ij")
    out[offset(r, kb, l, rows, blocks).ravel()] = sf.ravel()
    return out


def unpack(buf: np.ndarray, rows: int, blocks: int, batch: int = 1) -> np.ndarray:
    """Flat physical uint8 buffer -> logical (batch, rows, blocks) scale bytes."""
    buf = np.asarray(buf, dtype=np.uint8).ravel()
    l, r, kb = np.meshgrid(np.arange(batch), np.arange(rows), np.arange(blocks), indexing="ij")
    return buf[offset(r, kb, l, rows, blocks)]


def unpack_rows(buf: np.ndarray, row_ids, blocks: int, rows: int, batch_of_row=None) -> np.ndarray:
    """Scale bytes (len(row_ids), blocks) of selected rows (flat ids l*rows + r when batched)."""
    row_ids = np.asarray(row_ids, dtype=np.int64)
    l = row_ids // rows if batch_of_row is None else np.asarray(batch_of_row)
    r = row_ids % rows
    kb = np.arange(blocks)
    return np.asarray(buf, dtype=np.uint8).ravel()[offset(r[:, None], kb[None, :], l[:, None], rows, blocks)]

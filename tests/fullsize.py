"""Oracle side of the full-size parity tests: the workloads' operands run through the oracle's
quantiser row chunk by row chunk on host threads (rows are independent, and numpy releases the
interpreter lock inside its array operations), compared bit for bit with the GPU's codes and
scale bytes, and dequantised to float64.  The oracle functions are called unchanged; only the
split into row chunks and the threads are added here."""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

from oracle import quantize as oq, sf_layout

CHUNK_ROWS = 256
_POOL = cf.ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1)))


def tmap(fn, items):
    """fn over items on the host threads, in order."""
    return list(_POOL.map(fn, list(items)))


def row_chunks(r0: int, r1: int, step: int = CHUNK_ROWS):
    return [(a, min(a + step, r1)) for a in range(r0, r1, step)]


def checked_operand(x_fn, r0: int, r1: int, q_rows_gpu: np.ndarray, sf_gpu: np.ndarray, rows_per_batch: int,
                    fmt: str, k: int, what: str) -> np.ndarray:
    """Float64 values (r1 - r0, K) of flat operand rows [r0, r1) by the oracle, after checking that
    the GPU's codes (q_rows_gpu, the same rows) and scale bytes (the whole physical buffer
    sf_gpu) equal the oracle's.  x_fn(ids) returns the fp32 rows of flat ids."""
    v = 32 if fmt == "mxfp8" else 16
    out = np.empty((r1 - r0, k), dtype=np.float64)

    def one(span):
        a, b = span
        ids = np.arange(a, b)
        codes, sf_log = oq.quantize_logical(x_fn(ids)[None], fmt)
        if not np.array_equal(q_rows_gpu[a - r0:b - r0], codes[0]):
            return f"{what}: operand codes of rows {a}..{b - 1} differ from the oracle's"
        sf = sf_layout.unpack_rows(sf_gpu, ids, k // v, rows_per_batch)
        if not np.array_equal(sf, sf_log[0]):
            return f"{what}: operand scale bytes of rows {a}..{b - 1} differ from the oracle's"
        vals = oq.decode_codes(codes[0], fmt)
        out[a - r0:b - r0] = vals * np.repeat(oq.decode_scales(sf_log[0], fmt), v, axis=-1)
        return None

    errs = [e for e in tmap(one, row_chunks(r0, r1)) if e]
    assert not errs, errs[0]
    return out


def run_checks(fn, r: int, step: int = CHUNK_ROWS):
    """fn(a, b) over row chunks [a, b) of [0, r) on the host threads; returns their results."""
    return tmap(lambda span: fn(*span), row_chunks(0, r, step))

"""Row-chunked calls of the oracle on many host threads (test infrastructure).

The oracle's functions are pure and reentrant C, and ctypes releases the GIL
while they run, so disjoint row ranges of a full-size matrix can go through
the oracle at once on every host core.  Each chunk is the oracle's own
computation on those rows, unchanged: the per-row arithmetic and its order
are exactly those of a single call over the whole matrix.
"""
from __future__ import annotations

import concurrent.futures
import os

import numpy as np

THREADS = max(1, min(64, os.cpu_count() or 1))


def row_ranges(rows: int, parts: int | None = None):
    parts = max(1, min(rows, parts or 4 * THREADS))
    return [(rows * i // parts, rows * (i + 1) // parts) for i in range(parts)]


def par_map(fn, items):
    with concurrent.futures.ThreadPoolExecutor(THREADS) as ex:
        return list(ex.map(fn, items))


def prune_pack(orc, W: np.ndarray, N: int, M: int):
    """orc.prune_pack over every row of W [rows][cols] -> (values, masks)."""
    parts = par_map(lambda r: orc.prune_pack(W[r[0]:r[1]], N, M), row_ranges(W.shape[0]))
    return (np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]))


def spmv(orc, values: np.ndarray, masks: np.ndarray, cols: int, x: np.ndarray):
    """orc.spmv_f64 over every row of a packed matrix -> (y, s)."""
    parts = par_map(lambda r: orc.spmv_f64(values[r[0]:r[1]], masks[r[0]:r[1]], cols, x),
                    row_ranges(masks.shape[0]))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def matvec(orc, W: np.ndarray, x: np.ndarray):
    """orc.matvec_f64 over every row of a dense matrix -> (y, s)."""
    parts = par_map(lambda r: orc.matvec_f64(W[r[0]:r[1]], x), row_ranges(W.shape[0]))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def spmv_tokens(orc, values: np.ndarray, masks: np.ndarray, cols: int, X: np.ndarray):
    """orc.spmv_f64 of every token X[t] over every row -> (Y [T][rows], S [T][rows])."""
    parts = par_map(lambda t: orc.spmv_f64(values, masks, cols, X[t]), range(X.shape[0]))
    return np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts])

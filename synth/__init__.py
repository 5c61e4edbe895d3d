"""Seeded synthetic inputs shared by the tests and the benchmark.

This module draws numbers and nothing else: it holds none of the SpMV method's
arithmetic (no pruning, packing or products), so both the CUDA path and the
oracle can consume what it produces without sharing any of the method's code.

Recipe (the shapes and distributions of the SparseDecoding workloads):
  * weights: i.i.d. N(0, sigma=0.02), rounded to fp16 (round to nearest even);
  * activations x: i.i.d. N(0, 1), rounded to fp16;
  * exact-arithmetic inputs: w = k * 2^-6 with |k| <= 8, x integer in [-2, 2].
Every tensor is a pure function of (seed, stream id, element index) --
SplitMix64 in counter mode -- so any slice of any tensor can be regenerated
alone.  See ``synth.c`` for the published definitions used.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")

WEIGHT_SIGMA = 0.02
X_SIGMA = 1.0


def build(quiet: bool = True) -> str:
    cmd = ["gcc", "-std=gnu11", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
           "-Wall", _SRC, "-o", _LIB_PATH, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("synth build failed:\n" + res.stderr)
    return _LIB_PATH


_lib: ctypes.CDLL | None = None


def _load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            build()
        lib = ctypes.CDLL(_LIB_PATH)
        u64, i64, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        lib.synth_normal_f16.argtypes = [u64, u64, ctypes.c_double, i64, i64, p]
        lib.synth_normal_f16.restype = None
        lib.synth_int_f16.argtypes = [u64, u64, ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, i64, p]
        lib.synth_int_f16.restype = None
        lib.synth_u64.argtypes = [u64, u64, i64, i64, p]
        lib.synth_u64.restype = None
        _lib = lib
    return _lib


def stream_id(*parts: int) -> int:
    """Fold small non-negative integers (config, matrix, slot, role...) into one stream id."""
    sid = 0
    for p in parts:
        sid = (sid * 1_000_003 + int(p) + 1) & 0xFFFFFFFFFFFFFFFF
    return sid


def normal_f16_into(ptr: int, n: int, seed: int, stream: int, sigma: float, offset: int = 0) -> None:
    """Fill n fp16 bit patterns at host address ``ptr`` (e.g. a pinned tensor)."""
    _load().synth_normal_f16(seed, stream, float(sigma), offset, n, ptr)


def normal_f16(shape, seed: int, stream: int, sigma: float, offset: int = 0) -> np.ndarray:
    """N(0, sigma) rounded to fp16; returns uint16 bit patterns of ``shape``."""
    out = np.empty(shape, dtype=np.uint16)
    normal_f16_into(out.ctypes.data, out.size, seed, stream, sigma, offset)
    return out


def int_f16(shape, seed: int, stream: int, lo: int, hi: int, pow2: int = 0) -> np.ndarray:
    """Uniform integers k in [lo, hi] times 2^pow2, as exact fp16 bit patterns."""
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_int_f16(seed, stream, int(lo), int(hi), int(pow2), 0, out.size, out.ctypes.data)
    return out


def u64(n: int, seed: int, stream: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().synth_u64(seed, stream, 0, n, out.ctypes.data)
    return out


def weights(rows: int, cols: int, seed: int, stream: int) -> np.ndarray:
    return normal_f16((rows, cols), seed, stream, WEIGHT_SIGMA)


def activations(cols: int, seed: int, stream: int) -> np.ndarray:
    return normal_f16((cols,), seed, stream, X_SIGMA)


def sample_rows(rows: int, n: int, seed: int, stream: int) -> np.ndarray:
    """n distinct row indices in [0, rows), always including the first and last row."""
    n = min(n, rows)
    if n == rows:
        return np.arange(rows, dtype=np.int64)
    picks = {0, rows - 1}
    draws = u64(4 * n + 8, seed, stream)
    for d in draws:
        if len(picks) >= n:
            break
        picks.add(int(d % np.uint64(rows)))
    return np.array(sorted(picks), dtype=np.int64)

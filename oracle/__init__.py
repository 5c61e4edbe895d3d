"""Plain CPU oracle for batch-one N:M bitmask SpMV -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never loads it, and it shares
no code with the CUDA library: ``oracle.c`` is plain C99 in double precision,
compiled with ``gcc`` (no CUDA headers), and this file only marshals numpy
arrays into it.

What the oracle computes (SparseDecoding pages, see ``oracle.c``):
  * ``prune_pack``  -- dense fp16 -> compact values + one 32-bit mask word per
    32 input columns (aimodeling.com, "The Kernel Is the Other Half of the
    Answer"), the kept entries chosen as the N largest fp16 magnitudes of
    every M-group (synthetic pruner; ties to the lower column);
  * ``unpack``      -- the inverse scatter, unselected columns +0.0;
  * ``matvec_f64``  -- y = W x with double accumulation plus s = sum |w||x|;
  * ``spmv_rows_f64`` -- unpack + matvec for chosen rows of a packed matrix;
  * ``count_bad_words`` -- number of mask words whose popcount is not 16;
  * ``silu_mul_f64``  -- the SwiGLU epilogue silu(g) * u of a gate/up pair.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
against values fixed independently of this code (numpy's binary16, exact
rational arithmetic, brute-force subset enumeration, closed forms).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

# -ffp-contract=off: no fused multiply-add, so every double operation rounds
# exactly as written (and identically on x86-64 and aarch64).
CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-Wall", "-Wextra"]


def build(src: str = _SRC, out: str = _LIB_PATH, quiet: bool = True) -> str:
    """Compile ``oracle.c`` into a shared library with gcc; returns its path."""
    cmd = ["gcc", *CFLAGS, src, "-o", out, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + res.stderr)
    if not quiet and res.stderr:
        print(res.stderr)
    return out


_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.orc_f16_to_f64.restype = ctypes.c_double
    lib.orc_f16_from_f64.argtypes = [ctypes.c_double]
    lib.orc_f16_from_f64.restype = ctypes.c_uint16
    lib.orc_prune_pack.argtypes = [_P, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int, _P, _P]
    lib.orc_prune_pack.restype = ctypes.c_int
    lib.orc_unpack.argtypes = [_P, _P, _I64, _I64, _P, _I64]
    lib.orc_unpack.restype = ctypes.c_int
    lib.orc_matvec_f64.argtypes = [_P, _I64, _I64, _I64, _P, _P, _P]
    lib.orc_matvec_f64.restype = ctypes.c_int
    lib.orc_spmv_rows_f64.argtypes = [_P, _P, _I64, _I64, _P, _P, _I64, _P, _P]
    lib.orc_spmv_rows_f64.restype = ctypes.c_int
    lib.orc_count_bad_words.argtypes = [_P, _I64, _I64]
    lib.orc_count_bad_words.restype = ctypes.c_int64
    lib.orc_silu_mul_f64.argtypes = [_P, _P, _I64, _P]
    lib.orc_silu_mul_f64.restype = ctypes.c_int
    return lib


_lib: ctypes.CDLL | None = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if absent) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            build()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected fp16 bit patterns (uint16), got {a.dtype}")
    return a


class Oracle:
    """numpy-facing wrapper over one loaded copy of the oracle library."""

    def __init__(self, lib: ctypes.CDLL | None = None):
        self.lib = lib if lib is not None else load()

    # -- binary16 --------------------------------------------------------
    def f16_to_f64(self, h: int) -> float:
        return self.lib.orc_f16_to_f64(int(h))

    def f16_from_f64(self, v: float) -> int:
        return int(self.lib.orc_f16_from_f64(float(v)))

    # -- format ------------------------------------------------------------
    def prune_pack(self, W, N: int, M: int, cols: int | None = None):
        """W: [rows][ld] fp16 bits (first ``cols`` columns used, default all)
        -> (values [rows][cols/2] u16, masks [rows][cols/32] u32)."""
        W = _u16(W)
        rows, ld = W.shape
        cols = ld if cols is None else cols
        values = np.zeros((rows, cols // 2), dtype=np.uint16)
        masks = np.zeros((rows, max(cols // 32, 0)), dtype=np.uint32)
        rc = self.lib.orc_prune_pack(_ptr(W), rows, cols, ld, N, M, _ptr(values), _ptr(masks))
        if rc != 0:
            raise ValueError(f"orc_prune_pack rejected rows={rows} cols={cols} {N}:{M}")
        return values, masks

    def unpack(self, values, masks, cols: int) -> np.ndarray:
        values = _u16(values)
        masks = np.ascontiguousarray(masks, dtype=np.uint32)
        rows = masks.shape[0]
        W = np.zeros((rows, cols), dtype=np.uint16)
        rc = self.lib.orc_unpack(_ptr(values), _ptr(masks), rows, cols, _ptr(W), cols)
        if rc != 0:
            raise ValueError("orc_unpack rejected its input (bad shape or a mask word with popcount != 16)")
        return W

    def count_bad_words(self, masks, cols: int) -> int:
        masks = np.ascontiguousarray(masks, dtype=np.uint32)
        return int(self.lib.orc_count_bad_words(_ptr(masks), masks.shape[0], cols))

    # -- products ----------------------------------------------------------
    def matvec_f64(self, W, x, cols: int | None = None):
        """Dense y = W x in double over the first ``cols`` columns of W
        [rows][ld]; returns (y, s) with s = sum |w||x| per row."""
        W = _u16(W)
        x = _u16(x)
        rows, ld = W.shape
        cols = ld if cols is None else cols
        y = np.zeros(rows, dtype=np.float64)
        s = np.zeros(rows, dtype=np.float64)
        rc = self.lib.orc_matvec_f64(_ptr(W), rows, cols, ld, _ptr(x), _ptr(y), _ptr(s))
        if rc != 0:
            raise ValueError("orc_matvec_f64 rejected its input")
        return y, s

    def spmv_rows_f64(self, values, masks, cols: int, x, row_ids):
        """Packed y[row_ids] = (unpack(values, masks) x)[row_ids] in double; returns (y, s)."""
        values = _u16(values)
        masks = np.ascontiguousarray(masks, dtype=np.uint32)
        x = _u16(x)
        ids = np.ascontiguousarray(row_ids, dtype=np.int64)
        y = np.zeros(ids.shape[0], dtype=np.float64)
        s = np.zeros(ids.shape[0], dtype=np.float64)
        rc = self.lib.orc_spmv_rows_f64(_ptr(values), _ptr(masks), masks.shape[0], cols,
                                        _ptr(x), _ptr(ids), ids.shape[0], _ptr(y), _ptr(s))
        if rc != 0:
            raise ValueError("orc_spmv_rows_f64 rejected its input")
        return y, s

    def spmv_f64(self, values, masks, cols: int, x):
        rows = np.asarray(masks).shape[0]
        return self.spmv_rows_f64(values, masks, cols, x, np.arange(rows, dtype=np.int64))

    def silu_mul_f64(self, g, u) -> np.ndarray:
        """h = silu(g) * u in double (the SwiGLU epilogue)."""
        g = np.ascontiguousarray(g, dtype=np.float64)
        u = np.ascontiguousarray(u, dtype=np.float64)
        h = np.zeros_like(g)
        if self.lib.orc_silu_mul_f64(_ptr(g), _ptr(u), g.size, _ptr(h)) != 0:
            raise ValueError("orc_silu_mul_f64 rejected its input")
        return h

    def round_f16(self, y) -> np.ndarray:
        """Round doubles to binary16 bit patterns with the oracle's own RNE routine."""
        y = np.asarray(y, dtype=np.float64).ravel()
        return np.array([self.f16_from_f64(v) for v in y], dtype=np.uint16)


def tolerance(s: np.ndarray) -> np.ndarray:
    """Per-row acceptance bound for an fp16-output, fp32-accumulated SpMV:
    |y - y_ref| <= 2e-3 * sum|w||x| + 1e-5."""
    return 2e-3 * np.asarray(s, dtype=np.float64) + 1e-5

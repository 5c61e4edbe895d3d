"""Batch-one N:M bitmask SpMV for GB300 (sm_103a): Python binding.

A thin ctypes layer over ``libnmspmv.so`` (the C ABI in ``include/nm_spmv.h``).
It only marshals arguments: tensors become device pointers, the current
PyTorch stream becomes the ``cudaStream_t``, and output tensors are allocated
with PyTorch when the caller passes none.  Every step of the computation runs
in the library's CUDA kernels; there is no fallback path.  Importing works
without a GPU (so the symbol table can be checked), but the library itself
must exist: build it with ``__graft_entry__.build()`` or
``python -m sparse_spmv_memory_gb300._build``.

The operation (SparseDecoding, aimodeling.com article, "The Kernel Is the
Other Half of the Answer"): y = W x for one token, with W kept N:M-sparse
(2:4, 4:8, 8:16, 16:32) and stored as compact fp16 values plus one 32-bit
mask word per 32 input columns.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

__all__ = [
    "NMError", "lib", "library_path",
    "nm_status_string", "nm_values_bytes", "nm_masks_bytes", "nm_spmv_workspace_bytes",
    "nm_spmv_max_cols", "nm_pack", "nm_unpack", "nm_spmv", "nm_spmv_plan", "dense_gemv",
    "nm_check_masks", "nm_check_masks_noalloc", "nm_spmv_variant_count",
    "dense_gemv_variant_count", "nm_spmm", "nm_spmm_workspace_bytes", "nm_spmm_variant_count",
    "nm_spmm24", "nm_spmm24_workspace_bytes", "nm_spmm24_variant_count",
    "nm_spmv_swiglu", "nm_spmm_prefill", "nm_spmm_prefill_variant_count",
    "nm_spmm_prefill_workspace_bytes", "nm_spmm_prefill_plan", "nm_wait_timeouts",
    "nm_prefill_stall_selftest",
]

NM_OK = 0
NM_FLAG_PDL = 1
NM_FLAG_WEIGHTS_CONST = 2
STATUS_NAMES = {0: "NM_OK", 1: "NM_ERR_NULL", 2: "NM_ERR_SHAPE", 3: "NM_ERR_PATTERN",
                4: "NM_ERR_ALIGN", 5: "NM_ERR_WORKSPACE", 6: "NM_ERR_CUDA", 7: "NM_ERR_ALIAS"}


class NMError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {nm_status_string(status)}")


_lib: ctypes.CDLL | None = None


def library_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded C library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is missing: build it with __graft_entry__.build() "
                "(there is no CPU fallback)")
        _lib = _declare(ctypes.CDLL(path))
    return _lib


def _declare(L: ctypes.CDLL) -> ctypes.CDLL:
    P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    sig = {
        "nm_status_string": ([I32], ctypes.c_char_p),
        "nm_values_bytes": ([I64, I64], SZ),
        "nm_masks_bytes": ([I64, I64], SZ),
        "nm_spmv_workspace_bytes": ([I64, I64], SZ),
        "nm_spmv_max_cols": ([], I64),
        "nm_pack": ([P, I64, I64, I64, I32, I32, P, P, P], I32),
        "nm_unpack": ([P, P, I64, I64, P, I64, P], I32),
        "nm_spmv": ([P, P, I64, I64, P, P, P, SZ, P], I32),
        "nm_spmv_ex": ([P, P, I64, I64, P, P, P, SZ, I32, I32, I32, P], I32),
        "nm_spmv_plan": ([I64, I64, P, P, P], I32),
        "nm_spmv_variant_count": ([], I32),
        "dense_gemv": ([P, I64, I64, I64, P, P, P], I32),
        "dense_gemv_ex": ([P, I64, I64, I64, P, P, I32, I32, I32, P], I32),
        "dense_gemv_variant_count": ([], I32),
        "nm_check_masks": ([P, I64, I64, P], I64),
        "nm_check_masks_noalloc": ([P, I64, I64, P], I64),
        "nm_spmv_swiglu": ([P, P, I64, I64, P, P, P], I32),
        "nm_spmv_swiglu_ex": ([P, P, I64, I64, P, P, I32, I32, I32, P], I32),
        "nm_spmm_workspace_bytes": ([I64, I64, I32], SZ),
        "nm_spmm_workspace_bytes_ex": ([I64, I64, I32, I32, I32], SZ),
        "nm_spmm": ([P, P, I64, I64, P, I64, I32, P, I64, P, SZ, P], I32),
        "nm_spmm_ex": ([P, P, I64, I64, P, I64, I32, P, I64, P, SZ, I32, I32, I32, I32, P], I32),
        "nm_spmm_variant_count": ([], I32),
        "nm_spmm24_workspace_bytes": ([I64, I64, I32], SZ),
        "nm_spmm24_workspace_bytes_ex": ([I64, I64, I32, I32, I32], SZ),
        "nm_spmm24": ([P, P, I64, I64, P, I64, I32, P, I64, P, SZ, P], I32),
        "nm_spmm24_ex": ([P, P, I64, I64, P, I64, I32, P, I64, P, SZ, I32, I32, I32, P], I32),
        "nm_spmm24_variant_count": ([], I32),
        "nm_spmm_prefill": ([P, P, I64, I64, P, I64, I64, P, I64, P], I32),
        "nm_spmm_prefill_ex": ([P, P, I64, I64, P, I64, I64, P, I64, I32, I32, P, SZ, P], I32),
        "nm_spmm_prefill_ws": ([P, P, I64, I64, P, I64, I64, P, I64, P, SZ, P], I32),
        "nm_spmm_prefill_workspace_bytes": ([I64, I64, I64], SZ),
        "nm_spmm_prefill_workspace_bytes_ex": ([I64, I64, I64, I32, I32], SZ),
        "nm_spmm_prefill_plan": ([I64, I64, I64, I32, P, P, P], I32),
        "nm_spmm_prefill_variant_count": ([], I32),
        "nm_wait_timeouts": ([I32], I64),
        "nm_prefill_stall_selftest": ([P, P, I64, I64, P, I64, I64, P, I64, I64, P], I32),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    return L


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _stream(stream) -> int:
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("nm_* calls take CUDA tensors (there is no CPU path)")


def _check(status: int, what: str) -> None:
    if status != NM_OK:
        raise NMError(status, what)


# ---------------------------------------------------------------------------
# the C ABI, one Python function per entry point
# ---------------------------------------------------------------------------
def nm_status_string(status: int) -> str:
    return lib().nm_status_string(int(status)).decode()


def nm_values_bytes(rows: int, cols: int) -> int:
    return lib().nm_values_bytes(rows, cols)


def nm_masks_bytes(rows: int, cols: int) -> int:
    return lib().nm_masks_bytes(rows, cols)


def nm_spmv_workspace_bytes(rows: int, cols: int) -> int:
    return lib().nm_spmv_workspace_bytes(rows, cols)


def nm_spmv_max_cols() -> int:
    return lib().nm_spmv_max_cols()


def nm_spmv_variant_count() -> int:
    return lib().nm_spmv_variant_count()


def dense_gemv_variant_count() -> int:
    return lib().dense_gemv_variant_count()


def nm_spmv_plan(rows: int, cols: int) -> tuple[int, int, int]:
    v, g, w = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib().nm_spmv_plan(rows, cols, ctypes.byref(v), ctypes.byref(g), ctypes.byref(w)),
           "nm_spmv_plan")
    return v.value, g.value, w.value


def nm_pack(W, N: int, M: int, cols: int | None = None, values=None, masks=None, stream=None):
    """Prune dense fp16 W [rows][ld] (first ``cols`` columns) to N:M and pack it.
    Returns (values fp16 [rows][cols/2], masks int32 [rows][cols/32] holding uint32 bits)."""
    torch = _torch()
    _need_cuda(W)
    rows, ld = W.shape
    cols = ld if cols is None else cols
    if W.dtype != torch.float16 or W.stride(1) != 1:
        raise ValueError("W must be fp16 with unit column stride")
    if values is None:
        values = torch.empty((rows, cols // 2), dtype=torch.float16, device=W.device)
    if masks is None:
        masks = torch.empty((rows, cols // 32), dtype=torch.int32, device=W.device)
    _need_cuda(values, masks)
    _check(lib().nm_pack(_ptr(W), rows, cols, W.stride(0), N, M, _ptr(values), _ptr(masks),
                         _stream(stream)), "nm_pack")
    return values, masks


def nm_unpack(values, masks, cols: int, out=None, stream=None):
    """Scatter packed values back to dense fp16 [rows][cols] (+0.0 where unselected)."""
    torch = _torch()
    _need_cuda(values, masks)
    rows = masks.shape[0]
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.float16, device=values.device)
    _need_cuda(out)
    _check(lib().nm_unpack(_ptr(values), _ptr(masks), rows, cols, _ptr(out), out.stride(0),
                           _stream(stream)), "nm_unpack")
    return out


def nm_spmv(values, masks, x, y=None, workspace=None, stream=None, variant: int = -1,
            grid: int = 0, flags: int | None = None):
    """y = W x (fp16 out, fp32 accumulation) on the packed format.  ``variant``,
    ``grid`` and ``flags`` select nm_spmv_ex (defaults: the library's plan)."""
    torch = _torch()
    _need_cuda(values, masks, x)
    rows = masks.shape[0]
    cols = x.shape[0]
    if y is None:
        y = torch.empty((rows,), dtype=torch.float16, device=x.device)
    _need_cuda(y, workspace)
    L = lib()
    if workspace is None and variant < 0:
        need = L.nm_spmv_workspace_bytes(rows, cols)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if variant < 0 and grid <= 0 and flags is None:
        st = L.nm_spmv(_ptr(values), _ptr(masks), rows, cols, _ptr(x), _ptr(y), _ptr(workspace),
                       ws_bytes, _stream(stream))
    else:
        st = L.nm_spmv_ex(_ptr(values), _ptr(masks), rows, cols, _ptr(x), _ptr(y),
                          _ptr(workspace), ws_bytes, variant, grid,
                          NM_FLAG_PDL if flags is None else flags, _stream(stream))
    _check(st, "nm_spmv")
    return y


def nm_spmv_swiglu(values, masks, x, h=None, stream=None, variant: int = -1, grid: int = 0,
                   flags: int | None = None):
    """h = silu(W_gate x) * (W_up x), the packed matrix holding gate and up rows
    interleaved (row 2i gate, row 2i+1 up); h fp16 [rows / 2]."""
    torch = _torch()
    _need_cuda(values, masks, x)
    rows = masks.shape[0]
    cols = x.shape[0]
    if h is None:
        h = torch.empty((rows // 2,), dtype=torch.float16, device=x.device)
    _need_cuda(h)
    L = lib()
    if variant < 0 and grid <= 0 and flags is None:
        st = L.nm_spmv_swiglu(_ptr(values), _ptr(masks), rows, cols, _ptr(x), _ptr(h),
                              _stream(stream))
    else:
        st = L.nm_spmv_swiglu_ex(_ptr(values), _ptr(masks), rows, cols, _ptr(x), _ptr(h),
                                 variant, grid, NM_FLAG_PDL if flags is None else flags,
                                 _stream(stream))
    _check(st, "nm_spmv_swiglu")
    return h


def nm_spmm_workspace_bytes(rows: int, cols: int, batch: int) -> int:
    return lib().nm_spmm_workspace_bytes(rows, cols, batch)


def nm_spmm_variant_count() -> int:
    return lib().nm_spmm_variant_count()


def nm_spmm(values, masks, X, Y=None, workspace=None, stream=None, variant: int = -1,
            grid: int = 0, slices: int = 0, flags: int | None = None, cols: int | None = None):
    """Y = W X for a batch of tokens: X fp16 [batch][ldx] (first ``cols``
    columns used), Y fp16 [batch][ldy].  Batches of 1..8 run on the CUDA
    cores, larger ones on the tensor cores (nm_spmm_prefill).  A workspace of
    nm_spmm_workspace_bytes(...) bytes is allocated with PyTorch when needed
    and none is given."""
    torch = _torch()
    _need_cuda(values, masks, X)
    rows = masks.shape[0]
    batch, ldx = X.shape
    cols = ldx if cols is None else cols
    if X.stride(1) != 1 or (Y is not None and Y.stride(1) != 1):
        raise ValueError("X and Y must have unit column stride")
    if Y is None:
        Y = torch.empty((batch, rows), dtype=torch.float16, device=X.device)
    _need_cuda(Y, workspace)
    L = lib()
    if workspace is None:
        need = (L.nm_spmm_workspace_bytes_ex(rows, cols, batch, variant, slices) if batch <= 8
                else L.nm_spmm_workspace_bytes(rows, cols, batch))
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=X.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if variant < 0 and grid <= 0 and slices <= 0 and flags is None:
        st = L.nm_spmm(_ptr(values), _ptr(masks), rows, cols, _ptr(X), X.stride(0), batch,
                       _ptr(Y), Y.stride(0), _ptr(workspace), ws_bytes, _stream(stream))
    else:
        st = L.nm_spmm_ex(_ptr(values), _ptr(masks), rows, cols, _ptr(X), X.stride(0), batch,
                          _ptr(Y), Y.stride(0), _ptr(workspace), ws_bytes, variant, grid, slices,
                          NM_FLAG_PDL if flags is None else flags, _stream(stream))
    _check(st, "nm_spmm")
    return Y


def nm_spmm24_workspace_bytes(rows: int, cols: int, batch: int, variant: int = -1,
                              grid: int = 0) -> int:
    L = lib()
    if variant < 0 and grid <= 0:
        return L.nm_spmm24_workspace_bytes(rows, cols, batch)
    return L.nm_spmm24_workspace_bytes_ex(rows, cols, batch, variant, grid)


def nm_spmm24_variant_count() -> int:
    return lib().nm_spmm24_variant_count()


def nm_spmm24(values, masks, X, Y=None, workspace=None, stream=None, variant: int = -1,
              grid: int = 0, flags: int | None = None, cols: int | None = None):
    """Y = W X for 1..8 tokens of a 2:4 matrix on the tensor cores: X fp16
    [batch][ldx] (first ``cols`` columns used), Y fp16 [batch][ldy].  The
    workspace must be zero-filled before its first use (every call leaves it
    zero-filled); a zeroed one of nm_spmm24_workspace_bytes(...) bytes is
    allocated with PyTorch when none is given."""
    torch = _torch()
    _need_cuda(values, masks, X)
    rows = masks.shape[0]
    batch, ldx = X.shape
    cols = ldx if cols is None else cols
    if X.stride(1) != 1 or (Y is not None and Y.stride(1) != 1):
        raise ValueError("X and Y must have unit column stride")
    if Y is None:
        Y = torch.empty((batch, rows), dtype=torch.float16, device=X.device)
    _need_cuda(Y, workspace)
    L = lib()
    if workspace is None:
        need = nm_spmm24_workspace_bytes(rows, cols, batch, variant, grid)
        if need:
            workspace = torch.zeros(need, dtype=torch.uint8, device=X.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if variant < 0 and grid <= 0 and flags is None:
        st = L.nm_spmm24(_ptr(values), _ptr(masks), rows, cols, _ptr(X), X.stride(0), batch,
                         _ptr(Y), Y.stride(0), _ptr(workspace), ws_bytes, _stream(stream))
    else:
        st = L.nm_spmm24_ex(_ptr(values), _ptr(masks), rows, cols, _ptr(X), X.stride(0), batch,
                            _ptr(Y), Y.stride(0), _ptr(workspace), ws_bytes, variant, grid,
                            NM_FLAG_PDL if flags is None else flags, _stream(stream))
    _check(st, "nm_spmm24")
    return Y


def nm_spmm_prefill_variant_count() -> int:
    return lib().nm_spmm_prefill_variant_count()


def nm_spmm_prefill_workspace_bytes(rows: int, cols: int, T: int, variant: int = -1,
                                    splits: int = 0) -> int:
    """Bytes of workspace the prefill plan needs (0: no K split)."""
    L = lib()
    if variant < 0 and splits <= 0:
        return L.nm_spmm_prefill_workspace_bytes(rows, cols, T)
    return L.nm_spmm_prefill_workspace_bytes_ex(rows, cols, T, variant, splits)


def nm_spmm_prefill_plan(rows: int, cols: int, T: int, sms: int = 0) -> tuple[int, int, int]:
    """(kernel variant, K slices, tokens per block) nm_spmm_prefill_ws takes for
    this shape on a device with ``sms`` SMs (0: the current device)."""
    v, z, n = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib().nm_spmm_prefill_plan(rows, cols, T, sms, ctypes.byref(v), ctypes.byref(z),
                                      ctypes.byref(n)), "nm_spmm_prefill_plan")
    return v.value, z.value, n.value


def nm_spmm_prefill(values, masks, X, Y=None, workspace=None, stream=None, variant: int = -1,
                    splits: int = 0, cols: int | None = None):
    """Y = W X for a prefill-sized batch on the tensor cores: X fp16 [T][ldx]
    (first ``cols`` columns used), Y fp16 [T][ldy].  ``splits`` <= 0 lets the
    plan cut the rows' words into K slices when that fills more SMs (a
    workspace is then allocated with PyTorch unless one is given); 1 never
    splits."""
    torch = _torch()
    _need_cuda(values, masks, X)
    rows = masks.shape[0]
    T, ldx = X.shape
    cols = ldx if cols is None else cols
    if X.stride(1) != 1 or (Y is not None and Y.stride(1) != 1):
        raise ValueError("X and Y must have unit column stride")
    if Y is None:
        Y = torch.empty((T, rows), dtype=torch.float16, device=X.device)
    _need_cuda(Y, workspace)
    L = lib()
    if workspace is None and splits != 1:
        need = nm_spmm_prefill_workspace_bytes(rows, cols, T, variant, splits)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=X.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if variant < 0 and splits <= 0:
        st = L.nm_spmm_prefill_ws(_ptr(values), _ptr(masks), rows, cols, _ptr(X), X.stride(0), T,
                                  _ptr(Y), Y.stride(0), _ptr(workspace), ws_bytes,
                                  _stream(stream))
    elif variant < 0 and splits == 1:
        st = L.nm_spmm_prefill(_ptr(values), _ptr(masks), rows, cols, _ptr(X), X.stride(0), T,
                               _ptr(Y), Y.stride(0), _stream(stream))
    else:
        st = L.nm_spmm_prefill_ex(_ptr(values), _ptr(masks), rows, cols, _ptr(X), X.stride(0), T,
                                  _ptr(Y), Y.stride(0), variant, splits, _ptr(workspace),
                                  ws_bytes, _stream(stream))
    _check(st, "nm_spmm_prefill")
    return Y


def nm_prefill_stall_selftest(values, masks, X, Y, wait_limit_us: int, stream=None):
    """Launch the prefill kernel with its weight producer disabled (every
    bounded wait runs out; Y is left untouched).  Self-test of the wait path."""
    _need_cuda(values, masks, X, Y)
    T, ldx = X.shape
    _check(lib().nm_prefill_stall_selftest(_ptr(values), _ptr(masks), masks.shape[0], ldx,
                                           _ptr(X), X.stride(0), T, _ptr(Y), Y.stride(0),
                                           int(wait_limit_us), _stream(stream)),
           "nm_prefill_stall_selftest")


def nm_wait_timeouts(reset: bool = False) -> int:
    """How many bounded in-kernel waits gave up (0 in every correct run)."""
    r = lib().nm_wait_timeouts(1 if reset else 0)
    if r < 0:
        raise NMError(-r, "nm_wait_timeouts")
    return r


def dense_gemv(W, x, y=None, cols: int | None = None, stream=None, variant: int = -1,
               grid: int = 0, flags: int | None = None):
    """Dense baseline y = W x on fp16 W [rows][ld]."""
    torch = _torch()
    _need_cuda(W, x)
    rows, ld = W.shape
    cols = x.shape[0] if cols is None else cols
    if y is None:
        y = torch.empty((rows,), dtype=torch.float16, device=x.device)
    _need_cuda(y)
    L = lib()
    if variant < 0 and grid <= 0 and flags is None:
        st = L.dense_gemv(_ptr(W), rows, cols, W.stride(0), _ptr(x), _ptr(y), _stream(stream))
    else:
        st = L.dense_gemv_ex(_ptr(W), rows, cols, W.stride(0), _ptr(x), _ptr(y), variant, grid,
                             NM_FLAG_PDL if flags is None else flags, _stream(stream))
    _check(st, "dense_gemv")
    return y


def nm_check_masks(masks, cols: int, stream=None) -> int:
    """Number of mask words whose popcount is not 16 (host-synchronous)."""
    _need_cuda(masks)
    r = lib().nm_check_masks(_ptr(masks), masks.shape[0], cols, _stream(stream))
    if r < 0:
        raise NMError(-r, "nm_check_masks")
    return r


def nm_check_masks_noalloc(masks, cols: int, stream=None) -> int:
    """As nm_check_masks, for callers that must not allocate device memory:
    the scratch is a fixed array inside the library (limit: rows * cols / 32
    <= 67,108,864 words).  Calls overlapping on the GPU race on that array."""
    _need_cuda(masks)
    r = lib().nm_check_masks_noalloc(_ptr(masks), masks.shape[0], cols, _stream(stream))
    if r < 0:
        raise NMError(-r, "nm_check_masks_noalloc")
    return r

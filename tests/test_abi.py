"""The C-ABI library builds, loads and exports every symbol the header
declares; host-only entry points answer without a GPU."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = re.sub(r"^\s*#[^\n]*", "", text, flags=re.M)  # preprocessor lines
        names += re.findall(r"\b([A-Za-z_]\w*)\s*\([^;{}]*\)\s*;", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def library():
    from sparse_spmv_memory_gb300 import _build
    path = _build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["nm_pack", "nm_unpack", "nm_spmv", "dense_gemv", "nm_check_masks",
                     "nm_values_bytes", "nm_masks_bytes", "nm_spmv_workspace_bytes",
                     "nm_status_string"]:
        assert required in names


def test_library_exports_every_declared_symbol(library):
    missing = [n for n in declared_functions() if not hasattr(library, n)]
    assert not missing, missing


def test_binding_covers_every_symbol():
    import sparse_spmv_memory_gb300 as nm
    L = nm.lib()
    for n in declared_functions():
        f = getattr(L, n)
        assert f.restype is not None or f.argtypes is not None, n


def test_host_only_entry_points():
    import sparse_spmv_memory_gb300 as nm
    assert nm.nm_status_string(0) == "NM_OK"
    assert "PATTERN" in nm.nm_status_string(3)
    assert nm.nm_status_string(99) == "unknown nm_status"
    for rows, cols in [(4096, 4096), (57344, 8192), (8192, 28672), (1, 32)]:
        assert nm.nm_values_bytes(rows, cols) == rows * cols
        assert nm.nm_masks_bytes(rows, cols) == rows * cols // 8
    assert nm.nm_values_bytes(4, 48) == 0 and nm.nm_masks_bytes(-1, 32) == 0
    assert nm.nm_spmv_workspace_bytes(4096, 4096) == 0
    assert nm.nm_spmv_variant_count() >= 1 and nm.dense_gemv_variant_count() >= 1
    # explicit prefill plans are sized on the host: K slices of whole boxes of
    # four mask words, fp32 [slices][T][rows]
    assert nm.nm_spmm_prefill_workspace_bytes(8192, 8192, 64, 3, 2) == 2 * 64 * 8192 * 4
    assert nm.nm_spmm_prefill_workspace_bytes(300, 1056, 77, 1, 5) == 5 * 77 * 300 * 4  # 8,8,8,8,1
    assert nm.nm_spmm_prefill_workspace_bytes(300, 1056, 77, 1, 1) == 0
    assert nm.nm_spmm_prefill_workspace_bytes(64, 128, 16, 0, 8) == 0     # one box: no split
    assert nm.nm_spmm_prefill_workspace_bytes(300, 1056, 77, 1, 65) == 0  # beyond 64: refused


def test_library_has_no_oracle_dependency():
    """The CUDA library is built from csrc/ alone: no oracle source, header or
    symbol takes part in it."""
    from sparse_spmv_memory_gb300 import _build
    for src in _build._inputs():
        assert os.sep + "oracle" + os.sep not in src
        text = open(src).read()
        assert "oracle" not in text.lower(), src
    import sparse_spmv_memory_gb300 as nm
    assert not hasattr(nm.lib(), "orc_matvec_f64")


def test_oversize_shapes_are_refused_before_any_cuda_call():
    """Shapes whose word count would wrap an int64 (or exceed the scratch of
    the no-allocation check) are refused by the argument checks alone, so
    these calls never reach the GPU: no device is needed to run them."""
    import sparse_spmv_memory_gb300 as nm
    L = nm.lib()
    fake = 0x1000  # a 4-byte aligned, never dereferenced pointer
    # rows * (cols / 32) wraps negative without the guard
    wrap_rows, wrap_cols = 3 * 2**61 + 40_960_000, 64
    assert L.nm_check_masks_noalloc(fake, wrap_rows, wrap_cols, None) == -5
    assert L.nm_check_masks_noalloc(fake, 2**40, 2**40, None) == -5
    assert L.nm_check_masks_noalloc(fake, 1, (67108864 + 1) * 32, None) == -5
    assert L.nm_check_masks_noalloc(fake, 67108864 // 256 + 1, 256 * 32, None) == -5
    assert L.nm_check_masks(fake, wrap_rows, wrap_cols, None) == -2
    assert L.nm_check_masks(fake, 1024, 2**40, None) == -2
    # the prefill entry points bound cols so the word count fits an int
    assert nm.nm_spmm_prefill_workspace_bytes(128, 2**37, 64, 0, 1) == 0
    assert L.nm_spmm_prefill_plan(128, 2**37, 64, 152, None, None, None) == 2
    assert L.nm_spmm_prefill_plan(128, 8192, 64, 152, None, None, None) == 0


def test_spmm24_refusals_need_no_device():
    """nm_spmm24's argument checks run before any CUDA call: bad pointers,
    shapes and plans are refused on a machine without a GPU."""
    import sparse_spmv_memory_gb300 as nm
    L = nm.lib()
    v, m, x, y = 0x10000, 0x20000, 0x30000, 0x40000  # aligned, never dereferenced
    ok = (v, m, 64, 1024, x, 1024, 4, y, 64)

    def call(values=v, masks=m, rows=64, cols=1024, X=x, ldx=1024, batch=4, Y=y, ldy=64,
             variant=-1, grid=0):
        return L.nm_spmm24_ex(values, masks, rows, cols, X, ldx, batch, Y, ldy, None, 0,
                              variant, grid, 1, None)

    assert call(values=0) == 1 and call(Y=0) == 1
    assert call(cols=1056, ldx=1056) == 2          # cols % 128 != 0
    assert call(batch=0) == 2 and call(batch=9) == 2
    assert call(ldx=512) == 2 and call(ldy=8) == 2
    assert call(variant=nm.nm_spmm24_variant_count()) == 2
    assert call(grid=65537) == 2
    assert call(values=v + 16) == 4                # values must be 32-byte aligned
    assert call(X=x + 8) == 4 and call(ldx=1028) == 4
    assert call(rows=0) == 0                       # a no-op
    assert L.nm_spmm24(*ok, None, 0, None) != 2    # the shape itself is fine
    assert nm.nm_spmm24_workspace_bytes(64, 1056, 4) == 0
    assert nm.nm_spmm24_workspace_bytes(64, 1024, 9) == 0
    assert nm.nm_spmm24_variant_count() >= 1


def test_spmm24_refuses_unit_counts_beyond_32_bits():
    import sparse_spmv_memory_gb300 as nm
    L = nm.lib()
    v, m, x, y = 0x10000, 0x20000, 0x30000, 0x40000
    rows, cols = 2**30, 2**15  # 2^26 panels x 2^8 units = 2^34
    assert L.nm_spmm24_ex(v, m, rows, cols, x, cols, 2, y, rows, None, 0, -1, 0, 1, None) == 2
    assert nm.nm_spmm24_workspace_bytes(rows, cols, 2) == 0

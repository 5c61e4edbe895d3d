"""The prefill plan (kernel variant and K slices) is chosen on the host from
the shape and the SM count; nm_spmm_prefill_plan answers without a GPU when
the SM count is given.  Properties checked: the plan's slices are whole
four-word mask boxes and agree with the workspace the library asks for; a
device with one SM never splits (a split cannot fill more SMs there, it only
adds the combine); short prompts over matrices with few 128-row tiles split,
long prompts over the 70B-shaped layer do not; the partial sums stay within
the 256 MB bound."""
import numpy as np
import pytest

LAYER_70B = [(10240, 8192), (8192, 8192), (57344, 8192), (8192, 28672)]
GB300_SMS = 152


@pytest.fixture(scope="module")
def nm():
    from sparse_spmv_memory_gb300 import _build
    _build.build()
    import sparse_spmv_memory_gb300 as m
    return m


def slices_of(words, splits):
    """Slice count of a split request: ceil(words / splits) words per slice,
    rounded up to whole boxes of four words."""
    if splits <= 1 or words <= 4:
        return 1
    per = -(-words // splits)
    per = min(words, -(-per // 4) * 4)
    return -(-words // per)


def test_plan_is_whole_boxes_and_matches_the_workspace(nm):
    rng = np.random.default_rng(5)
    for _ in range(300):
        rows = int(rng.integers(1, 60000))
        cols = 32 * int(rng.integers(1, 1000))
        T = int(rng.integers(1, 4096))
        sms = int(rng.choice([1, 8, 76, 132, 152, 304]))
        v, z, tokens = nm.nm_spmm_prefill_plan(rows, cols, T, sms)
        assert 0 <= v < nm.nm_spmm_prefill_variant_count()
        assert tokens in (64, 128, 256, 512)
        assert 1 <= z <= 8
        assert slices_of(cols // 32, z) == z
        ws = nm.nm_spmm_prefill_workspace_bytes(rows, cols, T, v, z)
        assert ws == (z * T * rows * 4 if z > 1 else 0)
        assert ws <= 256 << 20


def test_one_sm_never_splits(nm):
    for rows, cols in LAYER_70B + [(128, 4096), (300, 1056)]:
        for T in (1, 16, 64, 256, 2048):
            assert nm.nm_spmm_prefill_plan(rows, cols, T, 1)[1] == 1


def test_few_row_tiles_split_and_long_prompts_do_not(nm):
    plans = {(r, c, T): nm.nm_spmm_prefill_plan(r, c, T, GB300_SMS)
             for r, c in LAYER_70B for T in (64, 2048)}
    # 64 tokens: 80, 64 and 64 row tiles leave most of 152 SMs idle unsplit
    for r, c in [(10240, 8192), (8192, 8192), (8192, 28672)]:
        assert plans[(r, c, 64)][1] > 1, (r, c)
    # the 448 row tiles of gate+up already fill the SMs
    assert plans[(57344, 8192, 64)][1] == 1
    # 2048 tokens: four 512-token tiles per row tile, no split, largest token tile
    for r, c in LAYER_70B:
        assert plans[(r, c, 2048)] == (4, 1, 512), (r, c)
    assert nm.nm_spmm_prefill_plan(1024, 8192, 64, GB300_SMS)[1] > 1


def test_plan_refuses_bad_shapes(nm):
    import ctypes
    L = nm.lib()
    v, z = ctypes.c_int(), ctypes.c_int()
    for rows, cols, T in [(0, 64, 8), (64, 48, 8), (64, 64, 0), (-1, 64, 8)]:
        assert L.nm_spmm_prefill_plan(rows, cols, T, 152, ctypes.byref(v), ctypes.byref(z),
                                      None) == 2

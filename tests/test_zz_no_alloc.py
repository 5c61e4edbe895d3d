"""nm_check_masks_noalloc: the mask check for callers that must not allocate
device memory while they run (for instance a serving process that gave all
device memory to its own allocator at start-up).  Its scratch is a fixed
array inside the library, so it is checked here against the allocating
nm_check_masks, through the C ABI, on two calls in a row -- the second call
must not see anything left over from the first.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test; it also passes on its own in a
fresh process (the fixture builds and loads the library itself)."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_spmv_memory_gb300 import _build
    _build.build()
    import sparse_spmv_memory_gb300 as nm
    return nm.lib()


def masks_with_bad_words(rows, cols, bad_positions, seed):
    W = synth.weights(rows, cols, seed, synth.stream_id(30, rows, cols))
    _, m = oracle.Oracle().prune_pack(W, 4, 8)
    m = m.copy()
    flat = m.reshape(-1)
    for k, pos in enumerate(bad_positions):
        flat[pos] = [0x0, 0xFFFFFFFF, 0x1, 0x7FFF][k % 4]  # popcount 0, 32, 1, 15
    return torch.from_numpy(m.view(np.int32)).cuda()


def test_matches_allocating_check_two_calls_in_a_row(lib):
    s = torch.cuda.current_stream().cuda_stream
    # first call: 9 bad words spread over several 16384-word blocks
    rows, cols = 3000, 8192          # 768,000 words -> 47 blocks
    words = rows * cols // 32
    bad = sorted({int(v % words) for v in synth.u64(9, 0, synth.stream_id(31, 1))} | {0, words - 1})
    m1 = masks_with_bad_words(rows, cols, bad, 1)
    ref1 = lib.nm_check_masks(m1.data_ptr(), rows, cols, s)
    got1 = lib.nm_check_masks_noalloc(m1.data_ptr(), rows, cols, s)
    assert ref1 == len(bad) and got1 == ref1
    # second call, smaller input and no bad words: nothing may carry over
    rows2, cols2 = 700, 4096
    m2 = masks_with_bad_words(rows2, cols2, [], 2)
    ref2 = lib.nm_check_masks(m2.data_ptr(), rows2, cols2, s)
    got2 = lib.nm_check_masks_noalloc(m2.data_ptr(), rows2, cols2, s)
    assert ref2 == 0 and got2 == ref2
    # and once more on the first input
    assert lib.nm_check_masks_noalloc(m1.data_ptr(), rows, cols, s) == ref1


def test_rejects_inputs_beyond_the_scratch_limit(lib):
    s = torch.cuda.current_stream().cuda_stream
    m = masks_with_bad_words(32, 1024, [], 3)
    max_words = 67108864
    # rows * cols / 32 one block past the limit: rejected on the host, nothing launched
    assert lib.nm_check_masks_noalloc(m.data_ptr(), max_words // 32 + 512, 1024, s) == -5
    assert lib.nm_check_masks_noalloc(None, 32, 1024, s) == -1
    assert lib.nm_check_masks_noalloc(m.data_ptr(), 32, 1000, s) == -2
    assert lib.nm_check_masks_noalloc(m.data_ptr(), 0, 1024, s) == 0

"""GPU parity of the small-batch SpMM (Y = W X, 1..8 tokens) against the CPU
oracle: every column of Y is an SpMV, so the oracle's packed SpMV of each
token is the reference.  Within the stated tolerance on random inputs; bit
for bit on exact-arithmetic inputs for every kernel variant, column-slice
count and grid size."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from gpu_util import f16_to_f64, from_dev, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def nm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_spmv_memory_gb300 import _build
    _build.build()
    import sparse_spmv_memory_gb300 as m
    m.lib()
    return m


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


def gen(rows, cols, batch, tag, exact=False):
    sw = synth.stream_id(40, tag, rows, cols, batch, 0)
    sx = synth.stream_id(40, tag, rows, cols, batch, 1)
    if exact:
        W = synth.int_f16((rows, cols), 0, sw, -8, 8, -6)
        X = synth.int_f16((batch, cols), 0, sx, -2, 2, 0)
    else:
        W = synth.weights(rows, cols, 0, sw)
        X = synth.normal_f16((batch, cols), 0, sx, synth.X_SIGMA)
    return W, X


def oracle_spmm(orc, ov, om, cols, X):
    ys, ss = [], []
    for j in range(X.shape[0]):
        y, s = orc.spmv_f64(ov, om, cols, X[j])
        ys.append(y)
        ss.append(s)
    return np.stack(ys), np.stack(ss)


def dev_masks(om):
    return torch.from_numpy(om.view(np.int32)).cuda()


@pytest.mark.parametrize("rows,cols", [(1, 32), (33, 1056), (300, 4096), (129, 14336), (64, 5120)])
@pytest.mark.parametrize("batch", [1, 2, 3, 5, 8])
def test_spmm_within_tolerance(nm, orc, rows, cols, batch):
    W, X = gen(rows, cols, batch, 1)
    N, M = [(2, 4), (4, 8), (8, 16), (16, 32)][batch % 4]
    ov, om = orc.prune_pack(W, N, M)
    Y = from_dev(nm.nm_spmm(to_dev(ov), dev_masks(om), to_dev(X)))
    ref, s = oracle_spmm(orc, ov, om, cols, X)
    err = np.abs(f16_to_f64(Y) - ref)
    assert np.all(err <= oracle.tolerance(s)), (rows, cols, batch, err.max())


@pytest.mark.parametrize("rows,cols", [(33, 1056), (300, 4096), (129, 14336)])
def test_spmm_exact_every_plan(nm, orc, rows, cols):
    """Exact sums: Y must equal the oracle's fp16 rounding bit for bit for every
    variant, column-slice count (partials summed by the second kernel) and grid."""
    T = (cols // 32 + 31) // 32
    for batch in (2, 4, 6, 7):
        W, X = gen(rows, cols, batch, 2, exact=True)
        ov, om = orc.prune_pack(W, 2, 4)
        ref, _ = oracle_spmm(orc, ov, om, cols, X)
        expect = np.stack([orc.round_f16(r) for r in ref])
        v, m, Xd = to_dev(ov), dev_masks(om), to_dev(X)
        L = nm.lib()
        for variant in range(nm.nm_spmm_variant_count()):
            # the fewest slices whose x tile fits this variant (more always may)
            ws = L.nm_spmm_workspace_bytes_ex(rows, cols, batch, variant, 0)
            s_min = ws // (batch * rows * 4) if ws else 1
            for slices in sorted({0, 1, min(2, T), min(3, T), T}):
                if 0 < slices < s_min:
                    with pytest.raises(nm.NMError) as e:
                        nm.nm_spmm(v, m, Xd, variant=variant, slices=slices)
                    assert e.value.status == 2  # does not fit: refused, nothing launched
                    continue
                for grid in (0, 7):
                    flags = (0, 1, 3)[(variant + slices + grid) % 3]
                    Y = nm.nm_spmm(v, m, Xd, variant=variant, grid=grid, slices=slices,
                                   flags=flags)
                    got = from_dev(Y)
                    assert np.array_equal(got, expect), (batch, variant, slices, grid)


def test_spmm_batch_one_equals_spmv_on_exact_inputs(nm, orc):
    rows, cols = 500, 8192
    W, X = gen(rows, cols, 1, 3, exact=True)
    v, m = nm.nm_pack(to_dev(W), 8, 16)
    Xd = to_dev(X)
    y1 = from_dev(nm.nm_spmv(v, m, Xd[0]))
    Y = from_dev(nm.nm_spmm(v, m, Xd))
    assert np.array_equal(Y[0], y1)


def test_spmm_strided_and_workspace(nm, orc):
    rows, cols, batch = 200, 2048, 6
    ldx, ldy = cols + 64, rows + 9
    Wf, Xw = gen(rows, ldx, batch, 4)
    W = np.ascontiguousarray(Wf[:, :cols])
    ov, om = orc.prune_pack(W, 4, 8)
    v, m = to_dev(ov), dev_masks(om)
    Xd = to_dev(Xw)
    Yd = torch.full((batch, ldy), 3.0, dtype=torch.float16, device="cuda")
    nm.nm_spmm(v, m, Xd, Y=Yd, cols=cols, slices=2)
    got = from_dev(Yd)
    ref, s = oracle_spmm(orc, ov, om, cols, np.ascontiguousarray(Xw[:, :cols]))
    assert np.all(np.abs(f16_to_f64(got[:, :rows]) - ref) <= oracle.tolerance(s))
    assert np.all(got[:, rows:] == np.float16(3.0).view(np.uint16))  # untouched
    # a slice plan needs the workspace: too small is refused before any launch
    L = nm.lib()
    s_ = torch.cuda.current_stream().cuda_stream
    st = L.nm_spmm_ex(v.data_ptr(), m.data_ptr(), rows, cols, Xd.data_ptr(), ldx, batch,
                      Yd.data_ptr(), ldy, None, 0, 0, 0, 2, 1, s_)
    assert st == 5
    assert L.nm_spmm_ex(v.data_ptr(), m.data_ptr(), rows, cols, Xd.data_ptr(), ldx, 9,
                        Yd.data_ptr(), ldy, None, 0, 0, 0, 1, 1, s_) == 2   # batch > 8


def test_spmm_long_rows_need_slices(nm):
    # batch 8 on the 70B down projection: the x tile of a whole row does not fit
    assert nm.nm_spmm_workspace_bytes(8192, 28672, 8) > 0
    assert nm.nm_spmm_workspace_bytes(8192, 8192, 2) == 0


@pytest.mark.parametrize("cols", [1024, 1056, 28672])
@pytest.mark.parametrize("batch", [2, 4, 8])
def test_spmm_corrupt_masks_stay_in_bounds(nm, orc, cols, batch):
    """Mask words with popcount != 16 break the precondition: the kernel must
    still read inside its arrays (a chain that runs out of set bits reads a
    zero pad row of the x tile), every other row stays exact, and
    nm_check_masks counts the bad words.  1024 columns take the whole-step
    kernel, 1056 the general one (a ragged last step), 28672 at 4 and 8
    tokens the column-sliced path."""
    rows = 64
    W, X = gen(rows, cols, batch, 5, exact=True)
    ov, om = orc.prune_pack(W, 2, 4)
    ref, _ = oracle_spmm(orc, ov, om, cols, X)
    expect = np.stack([orc.round_f16(r) for r in ref])
    bad = om.copy()
    bad[5, 0] = 0x0            # popcount 0: both chains run out at once
    bad[9, 3] = 0xFFFFFFFF     # popcount 32
    bad[20, 31] = 0x1          # popcount 1
    bad[41, cols // 32 - 1] = 0x80000000  # popcount 1, the word's last column
    m = dev_masks(bad)
    assert nm.nm_check_masks(m, cols) == 4
    Y = from_dev(nm.nm_spmm(to_dev(ov), m, to_dev(X)))
    good = np.setdiff1d(np.arange(rows), [5, 9, 20, 41])
    assert np.array_equal(Y[:, good], expect[:, good])


def test_spmm_randomised_shapes_bit_exact(nm, orc):
    """Seeded random shapes (any rows; columns a multiple of 1024 for half
    the cases, so the whole-step kernel runs, any multiple of 32 otherwise;
    1..8 tokens; all four patterns), every variant, the automatic and a
    random larger column-slice count, the default and a random grid,
    exact-arithmetic inputs: bit-exact against the oracle."""
    from gpu_util import PATTERNS
    draws = synth.u64(96, 0, synth.stream_id(43))
    L = nm.lib()
    for k in range(16):
        d = [int(x) for x in draws[6 * k: 6 * k + 6]]
        rows = 1 + d[0] % 700
        cols = 1024 * (1 + d[1] % 12) if k % 2 == 0 else 32 * (1 + d[1] % 400)
        batch = 1 + d[2] % 8
        N, M = PATTERNS[d[3] % 4]
        W, X = gen(rows, cols, batch, 200 + k, exact=True)
        ov, om = orc.prune_pack(W, N, M)
        ref, _ = oracle_spmm(orc, ov, om, cols, X)
        expect = np.stack([orc.round_f16(r) for r in ref])
        v, m, Xd = to_dev(ov), dev_masks(om), to_dev(X)
        T = (cols // 32 + 31) // 32
        for variant in range(nm.nm_spmm_variant_count()):
            ws = L.nm_spmm_workspace_bytes_ex(rows, cols, batch, variant, 0)
            s_min = ws // (batch * rows * 4) if ws else 1
            for slices in sorted({0, s_min + (d[4] + variant) % (T - s_min + 1)}):
                for grid in (0, 1 + (d[5] + variant) % 300):
                    got = from_dev(nm.nm_spmm(v, m, Xd, variant=variant, grid=grid,
                                              slices=slices))
                    bad = np.argwhere(got != expect)
                    assert bad.size == 0, (f"rows {rows} cols {cols} batch {batch} {N}:{M} "
                                           f"variant {variant} slices {slices} grid {grid}: "
                                           f"{len(bad)} mismatches, first {bad[:3].tolist()}")

"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Inputs come from the shared seeded generator; expected values come only from
the oracle.  Pack/unpack must be bit-exact; SpMV and the dense GEMV must meet
|y - y_ref| <= 2e-3 * sum|w||x| + 1e-5 per row, and be bit-exact where the
arithmetic is exact (small-integer inputs, unit vectors).
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import oracle
import synth
from gpu_util import PATTERNS, WORKLOADS, f16_to_f64, from_dev, to_dev

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


SMALL = [(1, 32), (3, 96), (33, 1056), (300, 1056), (257, 4096), (64, 5120), (1000, 2048),
         (129, 14336)]


def gen(rows, cols, tag, seed=0):
    W = synth.weights(rows, cols, seed, synth.stream_id(7, tag, rows, cols, 0))
    x = synth.activations(cols, seed, synth.stream_id(7, tag, rows, cols, 1))
    return W, x


def gen_exact(rows, cols, tag, seed=0):
    W = synth.int_f16((rows, cols), seed, synth.stream_id(8, tag, rows, cols, 0), -8, 8, -6)
    x = synth.int_f16((cols,), seed, synth.stream_id(8, tag, rows, cols, 1), -2, 2, 0)
    return W, x


def assert_within_tol(y_gpu, y_ref, s, what=""):
    err = np.abs(f16_to_f64(y_gpu) - y_ref)
    tol = oracle.tolerance(s)
    bad = np.nonzero(~(err <= tol))[0]
    assert bad.size == 0, f"{what}: {bad.size} rows out of tolerance, first {bad[:5]}, err {err[bad[:5]]}, tol {tol[bad[:5]]}"


# ---------------------------------------------------------------------------
# pack / unpack
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("rows,cols", SMALL)
@pytest.mark.parametrize("N,M", PATTERNS)
def test_pack_bit_exact(nm, orc, rows, cols, N, M):
    W, _ = gen(rows, cols, 1)
    v, m = nm.nm_pack(to_dev(W), N, M)
    ov, om = orc.prune_pack(W, N, M)
    assert np.array_equal(from_dev(m), om)
    assert np.array_equal(from_dev(v), ov)


def test_pack_special_values(nm, orc):
    """+-0, subnormals, ties, +-inf and NaN in every group position."""
    pool = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x3C00, 0xBC00, 0x7C00, 0xFC00, 0x7E00,
                     0xFD00, 0x3800], dtype=np.uint16)
    idx = synth.u64(96 * 256, 0, synth.stream_id(9, 1)) % np.uint64(len(pool))
    W = pool[idx.astype(np.int64)].reshape(96, 256)
    for N, M in PATTERNS:
        v, m = nm.nm_pack(to_dev(W), N, M)
        ov, om = orc.prune_pack(W, N, M)
        assert np.array_equal(from_dev(m), om) and np.array_equal(from_dev(v), ov), (N, M)


@pytest.mark.parametrize("ld", [1056 + 8, 1056 + 3])
def test_pack_leading_dimension(nm, orc, ld):
    rows, cols = 70, 1056
    Wide = synth.weights(rows, ld, 0, synth.stream_id(10, ld))
    full = to_dev(Wide)
    v, m = nm.nm_pack(full, 4, 8, cols=cols)
    ov, om = orc.prune_pack(Wide, 4, 8, cols=cols)
    assert np.array_equal(from_dev(m), om) and np.array_equal(from_dev(v), ov)


@pytest.mark.parametrize("rows,cols", [(3, 96), (300, 1056), (129, 14336)])
def test_unpack_bit_exact(nm, orc, rows, cols):
    W, _ = gen(rows, cols, 2)
    for N, M in PATTERNS:
        ov, om = orc.prune_pack(W, N, M)
        dense = nm.nm_unpack(to_dev(ov), torch.from_numpy(om.view(np.int32)).cuda(), cols)
        assert np.array_equal(from_dev(dense), orc.unpack(ov, om, cols))


def test_unpack_into_wider_rows(nm, orc):
    rows, cols, ld = 40, 512, 520
    W, _ = gen(rows, cols, 3)
    ov, om = orc.prune_pack(W, 2, 4)
    out = torch.full((rows, ld), 7.0, dtype=torch.float16, device="cuda")
    nm.nm_unpack(to_dev(ov), torch.from_numpy(om.view(np.int32)).cuda(), cols, out=out)
    got = from_dev(out)
    assert np.array_equal(got[:, :cols], orc.unpack(ov, om, cols))
    assert np.all(got[:, cols:] == np.float16(7.0).view(np.uint16))  # untouched


# ---------------------------------------------------------------------------
# SpMV
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("rows,cols", SMALL)
@pytest.mark.parametrize("N,M", PATTERNS)
def test_spmv_within_tolerance(nm, orc, rows, cols, N, M):
    W, x = gen(rows, cols, 4)
    v, m = nm.nm_pack(to_dev(W), N, M)
    y = nm.nm_spmv(v, m, to_dev(x))
    ov, om = orc.prune_pack(W, N, M)
    y_ref, s = orc.spmv_f64(ov, om, cols, x)
    assert_within_tol(from_dev(y), y_ref, s, f"{rows}x{cols} {N}:{M}")


@pytest.mark.parametrize("rows,cols", [(1, 32), (33, 1056), (300, 1056), (257, 4096), (129, 14336)])
def test_spmv_exact_arithmetic_every_plan(nm, orc, rows, cols):
    """Small-integer inputs: fp32 sums are exact in any order, so the fp16
    output must equal the oracle's rounding of the exact sum, bit for bit,
    for every kernel variant and many grid sizes (rows cut in many places),
    with x 32-byte aligned and with x only 16-byte aligned (the least the
    entry point accepts)."""
    W, x = gen_exact(rows, cols, 5)
    for N, M in [(2, 4), (16, 32)]:
        ov, om = orc.prune_pack(W, N, M)
        y_ref, _ = orc.spmv_f64(ov, om, cols, x)
        expect = orc.round_f16(y_ref)
        v, m = to_dev(ov), torch.from_numpy(om.view(np.int32)).cuda()
        xd = to_dev(x)
        xbuf = torch.zeros(cols + 8, dtype=torch.float16, device="cuda")
        xbuf[8:] = xd  # same dtype: a bit copy
        x16 = xbuf[8:]  # 16 bytes past a 32-byte aligned allocation
        assert xd.data_ptr() % 32 == 0 and x16.data_ptr() % 32 == 16
        for variant in range(nm.nm_spmv_variant_count()):
            for grid in sorted({1, 2, 7, 152, rows}):
                flags = (0, 1, 3)[(variant + grid) % 3]  # plain, PDL, PDL + early weights
                xin = x16 if (variant + grid) % 2 else xd
                y = nm.nm_spmv(v, m, xin, variant=variant, grid=grid, flags=flags)
                got = from_dev(y)
                bad = np.nonzero(got != expect)[0]
                assert bad.size == 0, (N, M, variant, grid, bad[:5], got[bad[:5]], expect[bad[:5]])


@pytest.mark.parametrize("rows,cols", [(300, 1056), (1000, 2048)])
def test_spmv_every_plan_within_tolerance(nm, orc, rows, cols):
    W, x = gen(rows, cols, 6)
    ov, om = orc.prune_pack(W, 8, 16)
    y_ref, s = orc.spmv_f64(ov, om, cols, x)
    v, m = to_dev(ov), torch.from_numpy(om.view(np.int32)).cuda()
    xd = to_dev(x)
    for variant in range(nm.nm_spmv_variant_count()):
        for grid in (1, 3, 64, 152, 1000):
            assert_within_tol(from_dev(nm.nm_spmv(v, m, xd, variant=variant, grid=grid)),
                              y_ref, s, f"variant {variant} grid {grid}")


def test_spmv_unit_vectors_exact(nm, orc):
    rows, cols = 200, 2048
    W, _ = gen(rows, cols, 7)
    for N, M in PATTERNS:
        ov, om = orc.prune_pack(W, N, M)
        dense = orc.unpack(ov, om, cols)
        v, m = to_dev(ov), torch.from_numpy(om.view(np.int32)).cuda()
        for j in (0, 1, 31, 32, 1000, 2047):
            x = np.zeros(cols, dtype=np.uint16)
            x[j] = 0x3C00
            y = from_dev(nm.nm_spmv(v, m, to_dev(x)))
            col = dense[:, j].copy()
            col[col == 0x8000] = 0x0000  # -0 * 1 + 0 accumulates to +0
            assert np.array_equal(y, col), (N, M, j)


def test_chained_calls_with_pdl(nm):
    """y of one call is x of the next, kernels back to back on one stream: with
    programmatic dependent launch (and early weight loads) every call must
    still see its predecessor's output -- the chain must match the plain one
    bit for bit.  (|y| stays O(1): the gains are ~0.9 sparse, ~1.3 dense.)"""
    n = 4096
    _, x = gen(n, n, 17)
    mats = [nm.nm_pack(to_dev(synth.weights(n, n, 0, synth.stream_id(17, i))), 2, 4)
            for i in range(4)]
    Wd = [to_dev(synth.weights(n, n, 0, synth.stream_id(18, i))) for i in range(3)]
    outs = {}
    for flags in (0, 1, 3):
        cur = to_dev(x)
        for rep in range(3):
            for v, m in mats:
                cur = nm.nm_spmv(v, m, cur, flags=flags)
            for Wi in Wd:
                cur = nm.dense_gemv(Wi, cur, flags=flags)
        got = from_dev(cur)
        assert np.all(np.isfinite(got.view(np.float16)))
        outs[flags] = got
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[3])


def test_spmv_deterministic(nm):
    rows, cols = 4096, 4096
    W, x = gen(rows, cols, 8)
    v, m = nm.nm_pack(to_dev(W), 2, 4)
    xd = to_dev(x)
    y1 = nm.nm_spmv(v, m, xd).clone()
    y2 = nm.nm_spmv(v, m, xd)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_pattern_nesting_gives_identical_format_and_output(nm, orc):
    """A 2:4 mask is a valid 4:8/8:16/16:32 mask: repacking a 2:4-pruned
    matrix (kept entries nonzero) under every larger M gives the same bytes
    and therefore the same y, bit for bit."""
    rows, cols = 512, 4096
    W, x = gen(rows, cols, 9)
    W[(W & 0x7FFF) == 0] = 0x3C00
    ov, om = orc.prune_pack(W, 2, 4)
    pruned = to_dev(orc.unpack(ov, om, cols))
    xd = to_dev(x)
    outs = []
    for N, M in PATTERNS:
        v, m = nm.nm_pack(pruned, N, M)
        assert np.array_equal(from_dev(v), ov) and np.array_equal(from_dev(m), om)
        outs.append(from_dev(nm.nm_spmv(v, m, xd)))
    assert all(np.array_equal(outs[0], o) for o in outs[1:])


def test_spmv_long_rows(nm, orc):
    """Up to nm_spmv_max_cols() a row's x tile fits one block and no workspace
    is needed; longer rows run column-sliced through a workspace, and an
    explicit single-block plan for them is refused."""
    cmax = nm.nm_spmv_max_cols()
    assert cmax >= 28672
    rows = 5
    for cols in (cmax, cmax + 32, 4 * cmax + 1024):
        W, x = gen(rows, cols, 10)
        v, m = nm.nm_pack(to_dev(W), 2, 4)
        ov, om = orc.prune_pack(W, 2, 4)
        y_ref, s = orc.spmv_f64(ov, om, cols, x)
        need = nm.nm_spmv_workspace_bytes(rows, cols)
        assert (need == 0) == (cols <= cmax)
        assert_within_tol(from_dev(nm.nm_spmv(v, m, to_dev(x))), y_ref, s, f"cols {cols}")
        if need:
            L = nm.lib()
            y = torch.empty(rows, dtype=torch.float16, device="cuda")
            st_ = torch.cuda.current_stream().cuda_stream
            xd = to_dev(x)
            assert L.nm_spmv(v.data_ptr(), m.data_ptr(), rows, cols, xd.data_ptr(), y.data_ptr(),
                             None, 0, st_) == 5          # workspace required
            assert L.nm_spmv_ex(v.data_ptr(), m.data_ptr(), rows, cols, xd.data_ptr(),
                                y.data_ptr(), None, 0, 0, 0, 1, st_) == 2   # single-block plan


def test_corrupt_masks_stay_in_bounds(nm, orc):
    """Words with popcount != 16 are a broken precondition: the kernel must
    still read only inside its arrays (every other row stays exact) and
    nm_check_masks must count them."""
    rows, cols = 64, 1024
    W, x = gen_exact(rows, cols, 11)
    ov, om = orc.prune_pack(W, 2, 4)
    y_ref, _ = orc.spmv_f64(ov, om, cols, x)
    expect = orc.round_f16(y_ref)
    bad = om.copy()
    bad[5, 0] = 0x0            # popcount 0
    bad[9, 3] = 0xFFFFFFFF     # popcount 32
    bad[20, 31] = 0x1          # popcount 1
    m = torch.from_numpy(bad.view(np.int32)).cuda()
    assert nm.nm_check_masks(m, cols) == 3
    y = from_dev(nm.nm_spmv(to_dev(ov), m, to_dev(x)))
    good = np.setdiff1d(np.arange(rows), [5, 9, 20])
    assert np.array_equal(y[good], expect[good])


def test_check_masks_on_packed_output(nm):
    W, _ = gen(1000, 2048, 12)
    for N, M in PATTERNS:
        _, m = nm.nm_pack(to_dev(W), N, M)
        assert nm.nm_check_masks(m, 2048) == 0


# ---------------------------------------------------------------------------
# dense baseline
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 96), (300, 1056), (257, 4096), (129, 14336), (17, 520)])
def test_dense_gemv_within_tolerance(nm, orc, rows, cols):
    W, x = gen(rows, cols, 13)
    y_ref, s = orc.matvec_f64(W, x)
    Wd, xd = to_dev(W), to_dev(x)
    for variant in range(nm.dense_gemv_variant_count()):
        for grid in sorted({1, 5, 152, rows}):
            y = nm.dense_gemv(Wd, xd, variant=variant, grid=grid)
            assert_within_tol(from_dev(y), y_ref, s, f"dense {rows}x{cols} v{variant} g{grid}")


def test_dense_gemv_exact_and_strided(nm, orc):
    rows, cols, ld = 150, 1024, 1040
    Wide = synth.int_f16((rows, ld), 0, synth.stream_id(14, 1), -8, 8, -6)
    x = synth.int_f16((cols,), 0, synth.stream_id(14, 2), -2, 2, 0)
    y_ref, _ = orc.matvec_f64(Wide, x, cols=cols)
    y = nm.dense_gemv(to_dev(Wide), to_dev(x), cols=cols)
    assert np.array_equal(from_dev(y), orc.round_f16(y_ref))


# ---------------------------------------------------------------------------
# argument errors: reported before any launch
# ---------------------------------------------------------------------------
def test_argument_errors(nm):
    L = nm.lib()
    s = torch.cuda.current_stream().cuda_stream
    rows, cols = 64, 256
    W, x = gen(rows, cols, 15)
    Wd, xd = to_dev(W), to_dev(x)
    v, m = nm.nm_pack(Wd, 2, 4)
    y = torch.empty(rows, dtype=torch.float16, device="cuda")
    P = lambda t: t.data_ptr()
    assert L.nm_spmv(None, P(m), rows, cols, P(xd), P(y), None, 0, s) == 1
    assert L.nm_spmv(P(v), P(m), rows, cols - 16, P(xd), P(y), None, 0, s) == 2
    assert L.nm_spmv(P(v), P(m), -1, cols, P(xd), P(y), None, 0, s) == 2
    assert L.nm_spmv(P(v) + 16, P(m), rows, cols, P(xd), P(y), None, 0, s) == 4
    assert L.nm_spmv(P(v), P(m), rows, cols, P(xd) + 8, P(y), None, 0, s) == 4
    assert L.nm_spmv(P(v), P(m), rows, cols, P(xd), P(xd), None, 0, s) == 7
    assert L.nm_spmv(P(v), P(m), 0, cols, P(xd), P(y), None, 0, s) == 0
    assert L.nm_spmv_ex(P(v), P(m), rows, cols, P(xd), P(y), None, 0, 99, 0, 1, s) == 2
    vv, mm = torch.empty_like(v), torch.empty_like(m)
    for N, M in [(1, 4), (2, 8), (3, 4), (32, 64)]:
        assert L.nm_pack(P(Wd), rows, cols, cols, N, M, P(vv), P(mm), s) == 3
    assert L.nm_pack(P(Wd), rows, cols, cols - 32, 2, 4, P(vv), P(mm), s) == 2
    assert L.nm_pack(P(Wd), rows, cols, cols, 2, 4, P(Wd), P(mm), s) == 7
    assert L.nm_pack(P(Wd), rows, cols, cols, 2, 4, P(vv) + 8, P(mm), s) == 4
    assert L.dense_gemv(P(Wd) + 2, rows, cols, cols, P(xd), P(y), s) == 4
    assert L.dense_gemv(P(Wd), rows, cols, cols, P(xd), P(Wd) + 64, s) == 7
    assert L.nm_check_masks(None, rows, cols, s) == -1
    with pytest.raises(ValueError):
        nm.nm_spmv(v.cpu(), m.cpu(), x_cpu := torch.zeros(cols, dtype=torch.float16))
    torch.cuda.synchronize()
    assert torch.equal(v, nm.nm_pack(Wd, 2, 4)[0])  # rejected calls wrote nothing

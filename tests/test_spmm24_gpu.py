"""GPU parity of the 2:4 small-batch SpMM on the tensor cores (nm_spmm24)
against the CPU oracle.  Every column of Y is an SpMV of the 2:4 packing, so
the oracle's packed SpMV of each token is the reference: within the stated
tolerance on random inputs, bit for bit on exact-arithmetic inputs for every
kernel variant, grid size and launch flag (panels cut between warps and
blocks at many places and summed by the warp that completes them, column
slices), one zero-filled workspace reused by every shape and plan, and every
output of two 70B decoder matrices at full size."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import oracle_threads as ot
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
    sw = synth.stream_id(45, tag, rows, cols, batch, 0)
    sx = synth.stream_id(45, tag, rows, cols, batch, 1)
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


@pytest.mark.parametrize("rows,cols", [(1, 128), (17, 256), (300, 4096), (129, 14336),
                                       (64, 5120), (1000, 1152)])
@pytest.mark.parametrize("batch", [1, 2, 3, 5, 8])
def test_spmm24_within_tolerance(nm, orc, rows, cols, batch):
    W, X = gen(rows, cols, batch, 1)
    ov, om = orc.prune_pack(W, 2, 4)
    Y = from_dev(nm.nm_spmm24(to_dev(ov), dev_masks(om), to_dev(X)))
    ref, s = oracle_spmm(orc, ov, om, cols, X)
    err = np.abs(f16_to_f64(Y) - ref)
    assert np.all(err <= oracle.tolerance(s)), (rows, cols, batch, err.max())


@pytest.mark.parametrize("rows,cols", [(17, 128), (300, 4096), (129, 14336), (1000, 1152)])
def test_spmm24_exact_every_plan(nm, orc, rows, cols):
    """Exact sums: Y equals the oracle's fp16 rounding bit for bit for every
    variant, several grids (1 block: no cut between blocks; 7 and 333: panels
    cut between warps of different blocks; more warps than units) and flags."""
    for batch in (1, 4, 6, 8):
        W, X = gen(rows, cols, batch, 2, exact=True)
        ov, om = orc.prune_pack(W, 2, 4)
        ref, _ = oracle_spmm(orc, ov, om, cols, X)
        expect = np.stack([orc.round_f16(r) for r in ref])
        v, m, Xd = to_dev(ov), dev_masks(om), to_dev(X)
        for variant in range(nm.nm_spmm24_variant_count()):
            for grid in (0, 1, 7, 333):
                flags = (0, 1, 3)[(variant + grid) % 3]
                got = from_dev(nm.nm_spmm24(v, m, Xd, variant=variant, grid=grid, flags=flags))
                assert np.array_equal(got, expect), (batch, variant, grid)


def test_spmm24_matches_nm_spmm_on_exact_inputs_and_repeats(nm, orc):
    rows, cols, batch = 777, 8192, 8
    W, X = gen(rows, cols, batch, 3, exact=True)
    v, m = nm.nm_pack(to_dev(W), 2, 4)
    Xd = to_dev(X)
    Y1 = from_dev(nm.nm_spmm(v, m, Xd))
    Y2 = from_dev(nm.nm_spmm24(v, m, Xd))
    assert np.array_equal(Y1, Y2)
    W, X = gen(rows, cols, batch, 4)
    v, m = nm.nm_pack(to_dev(W), 2, 4)
    Xd = to_dev(X)
    first = from_dev(nm.nm_spmm24(v, m, Xd))
    for _ in range(3):
        assert np.array_equal(from_dev(nm.nm_spmm24(v, m, Xd)), first)


def test_spmm24_strided_and_refusals(nm, orc):
    rows, cols, batch = 200, 2048, 7
    ldx, ldy = cols + 64, rows + 9
    Wf, Xw = gen(rows, ldx, batch, 5)
    W = np.ascontiguousarray(Wf[:, :cols])
    ov, om = orc.prune_pack(W, 2, 4)
    v, m = to_dev(ov), dev_masks(om)
    Xd = to_dev(Xw)
    Yd = torch.full((batch, ldy), 3.0, dtype=torch.float16, device="cuda")
    nm.nm_spmm24(v, m, Xd, Y=Yd, cols=cols)
    got = from_dev(Yd)
    ref, s = oracle_spmm(orc, ov, om, cols, np.ascontiguousarray(Xw[:, :cols]))
    assert np.all(np.abs(f16_to_f64(got[:, :rows]) - ref) <= oracle.tolerance(s))
    assert np.all(got[:, rows:] == np.float16(3.0).view(np.uint16))  # untouched
    L = nm.lib()
    s_ = torch.cuda.current_stream().cuda_stream
    need = nm.nm_spmm24_workspace_bytes(rows, cols, batch)
    assert need >= 1024
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    args = (v.data_ptr(), m.data_ptr(), rows, cols, Xd.data_ptr(), ldx, batch, Yd.data_ptr(), ldy)
    assert L.nm_spmm24(*args, None, 0, s_) == 5                      # no workspace
    assert L.nm_spmm24(*args, ws.data_ptr(), need - 16, s_) == 5     # short workspace
    assert L.nm_spmm24(*args, ws.data_ptr(), need, s_) == 0
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0  # left zero-filled for the next call
    bad_cols = (v.data_ptr(), m.data_ptr(), rows, cols - 32, Xd.data_ptr(), ldx, batch,
                Yd.data_ptr(), ldy)
    assert L.nm_spmm24(*bad_cols, ws.data_ptr(), need, s_) == 2      # cols % 128 != 0
    assert L.nm_spmm24_ex(*args, ws.data_ptr(), need, 99, 0, 1, s_) == 2   # no such variant
    torch.cuda.synchronize()


def test_spmm24_malformed_masks_stay_in_bounds(nm, orc):
    """Mask groups that do not hold exactly two set bits are decoded in bounds;
    the rows that keep valid masks are still exact."""
    rows, cols, batch = 96, 1024, 8
    W, X = gen(rows, cols, batch, 6, exact=True)
    ov, om = orc.prune_pack(W, 2, 4)
    ref, _ = oracle_spmm(orc, ov, om, cols, X)
    expect = np.stack([orc.round_f16(r) for r in ref])
    bad = om.copy()
    bad_rows = [0, 17, 95]
    bad[0, :] = 0xFFFFFFFF
    bad[17, 3] = 0
    bad[95, 31] = 0x7777EEEE
    for variant in range(nm.nm_spmm24_variant_count()):
        got = from_dev(nm.nm_spmm24(to_dev(ov), dev_masks(bad), to_dev(X), variant=variant))
        keep = np.setdiff1d(np.arange(rows), bad_rows)
        assert np.array_equal(got[:, keep], expect[:, keep]), variant
    torch.cuda.synchronize()


def test_spmm24_non_finite_x_reaches_only_its_token(nm, orc):
    """Pruned weights enter the products as +0, so an inf in token 2's x turns
    all of token 2's outputs non-finite; the other tokens are unaffected."""
    rows, cols, batch = 64, 512, 4
    W, X = gen(rows, cols, batch, 7, exact=True)
    ov, om = orc.prune_pack(W, 2, 4)
    ref, _ = oracle_spmm(orc, ov, om, cols, X)
    expect = np.stack([orc.round_f16(r) for r in ref])
    Xi = X.copy()
    Xi[2, 37] = np.float16(np.inf).view(np.uint16)
    got = from_dev(nm.nm_spmm24(to_dev(ov), dev_masks(om), to_dev(Xi)))
    assert not np.any(np.isfinite(f16_to_f64(got[2])))
    keep = [0, 1, 3]
    assert np.array_equal(got[keep], expect[keep])


@pytest.mark.parametrize("rows,cols,batch", [(10240, 8192, 8), (8192, 28672, 5)])
def test_every_output_of_a_2_4_spmm_at_full_size(nm, orc, rows, cols, batch):
    """The default plan at full size: the 70B qkv matrix at 8 tokens and the
    down projection (two column slices: every panel summed from partials) at 5
    tokens; every row and token against the oracle."""
    W = synth.weights(rows, cols, 0, synth.stream_id(46, rows, cols))
    X = synth.normal_f16((batch, cols), 0, synth.stream_id(47, rows, cols), synth.X_SIGMA)
    v, m = nm.nm_pack(to_dev(W), 2, 4)
    Y = from_dev(nm.nm_spmm24(v, m, to_dev(X)))
    del v, m
    ov, om = ot.prune_pack(orc, W, 2, 4)
    for j in range(batch):
        y_ref, s = ot.spmv(orc, ov, om, cols, X[j])
        err = np.abs(f16_to_f64(Y[j]) - y_ref)
        bad = np.nonzero(~(err <= oracle.tolerance(s)))[0]
        assert bad.size == 0, (j, bad[:4], err[bad][:4])
    torch.cuda.empty_cache()


def test_spmm24_one_workspace_serves_every_shape_and_plan(nm, orc):
    """One zero-filled workspace, reused by calls of different shapes (sliced
    and unsliced columns), variants and grids: every call is exact and leaves
    the workspace zero-filled."""
    shapes = [(300, 4096, 8), (97, 28672, 5), (1000, 1152, 3), (64, 16384, 8)]
    L = nm.lib()
    need = max(L.nm_spmm24_workspace_bytes_ex(r, c, b, v, g) for r, c, b in shapes
               for v in range(nm.nm_spmm24_variant_count()) for g in (0, 7, 333))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for rows, cols, batch in shapes:
        W, X = gen(rows, cols, batch, 8, exact=True)
        ov, om = orc.prune_pack(W, 2, 4)
        ref, _ = oracle_spmm(orc, ov, om, cols, X)
        expect = np.stack([orc.round_f16(r) for r in ref])
        v, m, Xd = to_dev(ov), dev_masks(om), to_dev(X)
        for variant in range(nm.nm_spmm24_variant_count()):
            for grid in (0, 7, 333):
                got = from_dev(nm.nm_spmm24(v, m, Xd, workspace=ws, variant=variant, grid=grid))
                assert np.array_equal(got, expect), (rows, cols, batch, variant, grid)
                assert int(ws.count_nonzero()) == 0, (rows, cols, variant, grid)

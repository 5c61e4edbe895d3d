"""GPU parity of the tensor-core prefill SpMM (nm_spmm_prefill: Y = W X for
T tokens) against the CPU oracle.  Every column of Y is an SpMV, so the
oracle's packed SpMV of each token is the reference.  Bit for bit on
exact-arithmetic inputs (every product and partial sum is a multiple of 2^-6
below 2^12, exact in the fp32 accumulator whatever the order) for every
kernel variant, on shapes with ragged row and token tails; within the SpMV
tolerance on random inputs for all four patterns; full-size decoder shapes
on sampled rows and tokens."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from gpu_util import PATTERNS, f16_to_f64, from_dev, to_dev

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
    m.nm_wait_timeouts(reset=True)
    return m


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


def gen(rows, cols, T, tag, exact=False):
    sw = synth.stream_id(70, tag, rows, cols, T, 0)
    sx = synth.stream_id(70, tag, rows, cols, T, 1)
    if exact:
        W = synth.int_f16((rows, cols), 0, sw, -8, 8, -6)
        X = synth.int_f16((T, cols), 0, sx, -2, 2, 0)
    else:
        W = synth.weights(rows, cols, 0, sw)
        X = synth.normal_f16((T, cols), 0, sx, synth.X_SIGMA)
    return W, X


def oracle_Y(orc, ov, om, cols, X):
    ys, ss = [], []
    for t in range(X.shape[0]):
        y, s = orc.spmv_f64(ov, om, cols, X[t])
        ys.append(y)
        ss.append(s)
    return np.stack(ys), np.stack(ss)


def dev_packed(orc, W, N, M):
    ov, om = orc.prune_pack(W, N, M)
    v = to_dev(ov)
    m = torch.from_numpy(om.view(np.int32)).cuda()
    return ov, om, v, m


EXACT_SHAPES = [(128, 32, 64), (300, 1056, 77), (257, 2048, 600), (1000, 1024, 513),
                (64, 4096, 9)]


@pytest.mark.parametrize("rows,cols,T", EXACT_SHAPES)
def test_prefill_exact_every_variant(nm, orc, rows, cols, T):
    W, X = gen(rows, cols, T, 1, exact=True)
    ov, om, v, m = dev_packed(orc, W, 2, 4)
    y_ref, _ = oracle_Y(orc, ov, om, cols, X)
    want = orc.round_f16(y_ref).reshape(y_ref.shape)
    Xd = to_dev(X)
    for variant in range(nm.nm_spmm_prefill_variant_count()):
        Y = from_dev(nm.nm_spmm_prefill(v, m, Xd, variant=variant))
        bad = np.argwhere(Y != want)
        assert bad.size == 0, f"variant {variant}: {len(bad)} mismatches, first (t, r) {bad[:4].tolist()}"
    assert nm.nm_wait_timeouts() == 0


@pytest.mark.parametrize("N,M", PATTERNS)
def test_prefill_within_tolerance(nm, orc, N, M):
    rows, cols, T = 640, 4096, 300
    W, X = gen(rows, cols, T, 2 + N)
    ov, om, v, m = dev_packed(orc, W, N, M)
    y_ref, s = oracle_Y(orc, ov, om, cols, X)
    Y = f16_to_f64(from_dev(nm.nm_spmm_prefill(v, m, to_dev(X))))
    err = np.abs(Y - y_ref)
    assert np.all(err <= oracle.tolerance(s)), float((err / oracle.tolerance(s)).max())
    assert nm.nm_wait_timeouts() == 0


def test_prefill_strided_and_deterministic(nm, orc):
    """X and Y with leading dimensions wider than cols / rows: only the
    addressed elements are read and written, and repeated calls agree."""
    rows, cols, T = 200, 2048, 130
    W, X = gen(rows, cols, T, 9, exact=True)
    ov, om, v, m = dev_packed(orc, W, 4, 8)
    y_ref, _ = oracle_Y(orc, ov, om, cols, X)
    Xw = torch.zeros((T, cols + 64), dtype=torch.float16, device="cuda")
    Xw[:, :cols] = to_dev(X)
    Yw = torch.full((T, rows + 40), -7.0, dtype=torch.float16, device="cuda")
    nm.nm_spmm_prefill(v, m, Xw, Y=Yw, cols=cols)
    got = from_dev(Yw[:, :rows].contiguous())
    assert np.array_equal(got, orc.round_f16(y_ref).reshape(y_ref.shape))
    assert bool((Yw[:, rows:] == -7.0).all())
    first = Yw.clone()
    nm.nm_spmm_prefill(v, m, Xw, Y=Yw, cols=cols)
    assert torch.equal(first.view(torch.int16), Yw.view(torch.int16))


def test_prefill_argument_errors(nm):
    L = nm.lib()
    v = torch.zeros(64 * 32, dtype=torch.float16, device="cuda")
    m = torch.zeros(64 * 2, dtype=torch.int32, device="cuda")
    X = torch.zeros((16, 64), dtype=torch.float16, device="cuda")
    Y = torch.zeros((16, 64), dtype=torch.float16, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    P = lambda t: t.data_ptr()
    assert L.nm_spmm_prefill(None, P(m), 64, 64, P(X), 64, 16, P(Y), 64, st) == 1
    assert L.nm_spmm_prefill(P(v), P(m), 64, 48, P(X), 64, 16, P(Y), 64, st) == 2   # cols % 32
    assert L.nm_spmm_prefill(P(v), P(m), 64, 64, P(X), 32, 16, P(Y), 64, st) == 2   # ldx < cols
    assert L.nm_spmm_prefill(P(v), P(m), 64, 64, P(X), 64, 16, P(Y), 32, st) == 2   # ldy < rows
    assert L.nm_spmm_prefill(P(v) + 2, P(m), 64, 64, P(X), 64, 16, P(Y), 64, st) == 4
    assert L.nm_spmm_prefill(P(v), P(m), 64, 64, P(X) + 2, 64, 16, P(Y), 64, st) == 4
    assert L.nm_spmm_prefill(P(v), P(m), 64, 64, P(X), 64, 16, P(X), 64, st) == 7   # Y aliases X
    assert L.nm_spmm_prefill_ex(P(v), P(m), 64, 64, P(X), 64, 16, P(Y), 64, 99, 1, None, 0,
                                st) == 2                                        # variant
    assert L.nm_spmm_prefill_ex(P(v), P(m), 64, 64, P(X), 64, 16, P(Y), 64, 3, 65, None, 0,
                                st) == 2                                        # splits > 64
    assert L.nm_spmm_prefill(P(v), P(m), 64, 64, P(X), 64, 0, P(Y), 64, st) == 0    # T == 0
    # a K split needs its workspace (256 columns = 8 words: two slices of four)
    v2 = torch.zeros(64 * 128, dtype=torch.float16, device="cuda")
    m2 = torch.zeros(64 * 8, dtype=torch.int32, device="cuda")
    X2 = torch.zeros((16, 256), dtype=torch.float16, device="cuda")
    need = L.nm_spmm_prefill_workspace_bytes_ex(64, 256, 16, 3, 2)
    assert need == 2 * 16 * 64 * 4
    ws = torch.zeros(need + 16, dtype=torch.uint8, device="cuda")
    args = (P(v2), P(m2), 64, 256, P(X2), 256, 16, P(Y), 64, 3, 2)
    assert L.nm_spmm_prefill_ex(*args, None, 0, st) == 5                       # no workspace
    assert L.nm_spmm_prefill_ex(*args, P(ws), need - 4, st) == 5              # short
    assert L.nm_spmm_prefill_ex(*args, P(ws) + 8, need, st) == 4              # misaligned
    assert L.nm_spmm_prefill_ex(*args, P(Y), need, st) == 7                   # aliases Y
    assert L.nm_spmm_prefill_ex(*args, P(ws), need, st) == 0
    torch.cuda.synchronize()


FULL = [(57344, 8192, 2048, (2, 4)), (10240, 8192, 1000, (16, 32)), (8192, 28672, 520, (8, 16)),
        (8192, 8192, 64, (2, 4)), (8192, 28672, 200, (4, 8))]


@pytest.mark.parametrize("rows,cols,T,pat", FULL)
def test_prefill_full_size_sampled(nm, orc, rows, cols, T, pat):
    """Decoder-layer shapes at prefill lengths, in the library's default plan
    (the short prompts on the 8192-row matrices take a K split): sampled rows
    (tile edges included) of sampled tokens (first and last included)
    against the oracle."""
    N, M = pat
    W = synth.weights(rows, cols, 0, synth.stream_id(71, rows, cols, 0))
    X = synth.normal_f16((T, cols), 0, synth.stream_id(71, rows, cols, 1), synth.X_SIGMA)
    Wd = to_dev(W)
    v, m = nm.nm_pack(Wd, N, M)
    del Wd
    Y = nm.nm_spmm_prefill(v, m, to_dev(X))
    torch.cuda.synchronize()
    assert nm.nm_wait_timeouts() == 0
    hv, hm = from_dev(v), from_dev(m)
    row_ids = np.unique(np.concatenate([
        synth.sample_rows(rows, 24, 0, synth.stream_id(72, rows)),
        np.array([127, 128, rows - 129, rows - 128], dtype=np.int64)]))
    toks = np.unique(np.concatenate([
        synth.sample_rows(T, 6, 0, synth.stream_id(73, T)),
        np.array([255, 256, 511, 512], dtype=np.int64)[np.array([255, 256, 511, 512]) < T]]))
    Yh = from_dev(Y)
    for t in toks:
        y_ref, s = orc.spmv_rows_f64(hv, hm, cols, X[t], row_ids)
        got = f16_to_f64(Yh[t, row_ids])
        assert np.all(np.abs(got - y_ref) <= oracle.tolerance(s)), f"token {t}"


def slices_of(words, splits):
    """Slice count the library derives from a split request: slices of
    ceil(words / splits) words rounded up to whole mask boxes of four."""
    if splits <= 1 or words <= 4:
        return 1
    per = -(-words // splits)              # ceil(words / splits)
    per = min(words, -(-per // 4) * 4)     # whole boxes of four words
    return -(-words // per)


SPLIT_SHAPES = [(300, 1056, 77), (257, 2048, 600), (64, 4096, 9), (128, 1024, 64), (200, 416, 130)]


@pytest.mark.parametrize("rows,cols,T", SPLIT_SHAPES)
def test_prefill_k_split_exact(nm, orc, rows, cols, T):
    """Explicit K splits for every variant -- slices of whole mask boxes, a
    ragged last slice, odd word counts (the cp.async mask path), up to one
    slice per box -- with the partial sums combined in slice order: bit-exact
    against the oracle on exact-arithmetic inputs, and repeatable."""
    W, X = gen(rows, cols, T, 14, exact=True)
    ov, om, v, m = dev_packed(orc, W, 2, 4)
    y_ref, _ = oracle_Y(orc, ov, om, cols, X)
    want = orc.round_f16(y_ref).reshape(y_ref.shape)
    Xd = to_dev(X)
    words = cols // 32
    for variant in range(nm.nm_spmm_prefill_variant_count()):
        for splits in sorted({2, 3, 5, min(words, 64)}):
            z = slices_of(words, splits)
            need = nm.nm_spmm_prefill_workspace_bytes(rows, cols, T, variant, splits)
            assert need == (z * T * rows * 4 if z > 1 else 0), (variant, splits)
            got = from_dev(nm.nm_spmm_prefill(v, m, Xd, variant=variant, splits=splits))
            bad = np.argwhere(got != want)
            assert bad.size == 0, (f"variant {variant} splits {splits} ({z} slices): "
                                   f"{len(bad)} mismatches, first {bad[:3].tolist()}")
    a = nm.nm_spmm_prefill(v, m, Xd, variant=3, splits=5)
    b = nm.nm_spmm_prefill(v, m, Xd, variant=3, splits=5)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert nm.nm_wait_timeouts() == 0


@pytest.mark.parametrize("N,M", PATTERNS)
def test_prefill_default_plan_splits_few_row_tiles(nm, orc, N, M):
    """Eight row tiles and 64 tokens fill few of the SMs: the default plan
    cuts K (it needs a workspace), and its result is within the tolerance of
    the oracle, like the unsplit call's."""
    rows, cols, T = 1024, 8192, 64
    assert nm.nm_spmm_prefill_workspace_bytes(rows, cols, T) > 0
    W, X = gen(rows, cols, T, 15 + N)
    ov, om, v, m = dev_packed(orc, W, N, M)
    y_ref, s = oracle_Y(orc, ov, om, cols, X)
    Xd = to_dev(X)
    for splits in (0, 1):
        Y = f16_to_f64(from_dev(nm.nm_spmm_prefill(v, m, Xd, splits=splits)))
        err = np.abs(Y - y_ref)
        assert np.all(err <= oracle.tolerance(s)), (splits, float((err / oracle.tolerance(s)).max()))
    assert nm.nm_wait_timeouts() == 0


def test_prefill_many_short_blocks_repeatable(nm, orc):
    """Tens of thousands of short blocks (eight K slices of 16 words on the
    512-token tile, 1792 blocks a call, 24 calls): every block's pipeline
    drains cleanly before the next block takes its SM, so no wait runs out
    and every call returns the same bits -- those of the unsplit call on
    exact-arithmetic inputs, and within the tolerance of the oracle on
    sampled rows."""
    rows, cols, T = 28672, 4096, 512
    W, X = gen(rows, cols, T, 16, exact=True)
    Wd = to_dev(W)
    v, m = nm.nm_pack(Wd, 2, 4)
    del Wd
    Xd = to_dev(X)
    ws = torch.empty(nm.nm_spmm_prefill_workspace_bytes(rows, cols, T, 4, 8), dtype=torch.uint8,
                     device="cuda")
    ref = nm.nm_spmm_prefill(v, m, Xd, variant=4, splits=1)
    Y = torch.empty_like(ref)
    nm.nm_wait_timeouts(reset=True)
    for _ in range(24):
        nm.nm_spmm_prefill(v, m, Xd, Y=Y, workspace=ws, variant=4, splits=8)
        assert torch.equal(Y.view(torch.int16), ref.view(torch.int16))
    assert nm.nm_wait_timeouts() == 0
    hv, hm = from_dev(v), from_dev(m)
    row_ids = np.array([0, 127, 128, 14335, rows - 1], dtype=np.int64)
    Yh = from_dev(Y)
    for t in (0, T - 1):
        y_ref, s = orc.spmv_rows_f64(hv, hm, cols, X[t], row_ids)
        assert np.all(np.abs(f16_to_f64(Yh[t, row_ids]) - y_ref) <= oracle.tolerance(s))


def test_prefill_every_plan_agrees_on_random_shapes(nm):
    """Seeded random shapes (both mask paths, all four patterns, ragged tiles)
    on exact-arithmetic inputs: every variant at 1, 2, 3, 5 and 8 K slices
    gives the same bits as the unsplit 64-token variant (itself checked
    against the oracle above), and no bounded wait runs out.  A soak of the
    barrier protocol under many short blocks and pipeline depths."""
    rng = np.random.default_rng(96)
    nm.nm_wait_timeouts(reset=True)
    done = 0
    while done < 400:
        rows = int(rng.integers(1, 1500))
        words = int(rng.integers(1, 96))
        T = int(rng.integers(1, 600))
        cols = 32 * words
        if rows * cols * T > 4e8:
            continue
        N, M = PATTERNS[done % 4]
        W = synth.int_f16((rows, cols), 0, synth.stream_id(96, done, 0), -8, 8, -6)
        X = synth.int_f16((T, cols), 0, synth.stream_id(96, done, 1), -2, 2, 0)
        Wd = to_dev(W)
        v, m = nm.nm_pack(Wd, N, M)
        del Wd
        Xd = to_dev(X)
        ref = nm.nm_spmm_prefill(v, m, Xd, variant=3, splits=1)
        for variant in range(nm.nm_spmm_prefill_variant_count()):
            for splits in (1, 2, 3, 5, 8):
                Y = nm.nm_spmm_prefill(v, m, Xd, variant=variant, splits=splits)
                assert torch.equal(Y.view(torch.int16), ref.view(torch.int16)), (
                    rows, cols, T, (N, M), variant, splits)
        done += 1
    assert nm.nm_wait_timeouts() == 0


def test_prefill_nonfinite_activation_is_dense_semantics(nm, orc):
    """Pruned weights enter the MMA as +0: an infinite X[t][c] makes every row
    that prunes column c NaN (0 * inf) and every row that keeps it +-inf (the
    sign of its weight); the other tokens are untouched."""
    rows, cols, T = 256, 1024, 64
    W, X = gen(rows, cols, T, 11)
    t_bad, c_bad = 5, 100
    X[t_bad, c_bad] = np.uint16(0x7C00)   # +inf
    ov, om, v, m = dev_packed(orc, W, 2, 4)
    Y = f16_to_f64(from_dev(nm.nm_spmm_prefill(v, m, to_dev(X))))
    kept = ((om[:, c_bad // 32] >> np.uint32(c_bad % 32)) & 1).astype(bool)
    Wp = f16_to_f64(orc.unpack(ov, om, cols))
    assert kept.any() and (~kept).any()
    assert np.isnan(Y[t_bad][~kept]).all()
    assert np.array_equal(np.sign(Y[t_bad][kept]), np.sign(Wp[kept, c_bad]))
    assert np.isinf(Y[t_bad][kept]).all()
    for t in range(T):
        if t == t_bad:
            continue
        y_ref, s = orc.spmv_f64(ov, om, cols, X[t])
        assert np.all(np.abs(Y[t] - y_ref) <= oracle.tolerance(s)), f"token {t}"


def test_nm_spmm_beyond_eight_tokens_takes_the_tensor_core_path(nm, orc):
    """nm_spmm with batch > 8 is served by the tensor-core path in its default
    plan (with the workspace nm_spmm_workspace_bytes names): the same bits."""
    rows, cols, T = 300, 2048, 12
    W, X = gen(rows, cols, T, 12)
    ov, om, v, m = dev_packed(orc, W, 8, 16)
    Xd = to_dev(X)
    a = from_dev(nm.nm_spmm(v, m, Xd))
    b = from_dev(nm.nm_spmm_prefill(v, m, Xd))
    assert np.array_equal(a, b)
    y_ref, s = oracle_Y(orc, ov, om, cols, X)
    assert np.all(np.abs(f16_to_f64(a) - y_ref) <= oracle.tolerance(s))


def test_nm_spmm_beyond_eight_tokens_asks_for_the_split_workspace(nm):
    """nm_spmm's workspace query covers the tensor-core plan beyond 8 tokens:
    a shape whose plan splits needs that workspace, and is refused without."""
    L = nm.lib()
    rows, cols, T = 1024, 8192, 64
    need = L.nm_spmm_workspace_bytes(rows, cols, T)
    assert need == nm.nm_spmm_prefill_workspace_bytes(rows, cols, T) > 0
    v = torch.zeros(rows * cols // 2, dtype=torch.float16, device="cuda")
    m = torch.zeros(rows * cols // 32, dtype=torch.int32, device="cuda")
    X = torch.zeros((T, cols), dtype=torch.float16, device="cuda")
    Y = torch.zeros((T, rows), dtype=torch.float16, device="cuda")
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    P = lambda t: t.data_ptr()
    args = (P(v), P(m), rows, cols, P(X), cols, T, P(Y), rows)
    assert L.nm_spmm(*args, None, 0, st) == 5
    assert L.nm_spmm(*args, P(ws), need - 16, st) == 5
    assert L.nm_spmm(*args, P(ws), need, st) == 0
    torch.cuda.synchronize()
    assert bool((Y == 0).all())     # all-zero weights: zero output
    assert nm.nm_wait_timeouts() == 0


def test_bounded_waits_end_a_stalled_prefill_kernel(nm, orc):
    """Self-test of the failure path: with its weight producer disabled no
    stage ever completes; every wait runs out after the given limit, is
    counted, the kernel stores nothing and returns, and the device stays
    usable for the next call (which is exact again)."""
    import time
    rows, cols, T = 256, 1024, 64
    W, X = gen(rows, cols, T, 13)
    ov, om, v, m = dev_packed(orc, W, 2, 4)
    Xd = to_dev(X)
    Y = torch.full((T, rows), 3.0, dtype=torch.float16, device="cuda")
    torch.cuda.synchronize()
    nm.nm_wait_timeouts(reset=True)
    t0 = time.time()
    nm.nm_prefill_stall_selftest(v, m, Xd, Y, wait_limit_us=20000)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert nm.nm_wait_timeouts(reset=True) > 0
    assert bool((Y == 3.0).all())
    # the first wait to give up aborts every other one: the launch ends after
    # about one wait limit (20 ms), not one per wait and block
    assert elapsed < 2.0
    Y2 = f16_to_f64(from_dev(nm.nm_spmm_prefill(v, m, Xd)))
    torch.cuda.synchronize()
    y_ref, s = oracle_Y(orc, ov, om, cols, X)
    assert np.all(np.abs(Y2 - y_ref) <= oracle.tolerance(s))
    assert nm.nm_wait_timeouts() == 0


def test_prefill_randomised_shapes_bit_exact(nm, orc):
    """Seeded random shapes (any rows, any multiple of 32 columns, any token
    count, all four patterns, odd and even word counts so both mask paths
    run), every variant, exact-arithmetic inputs: bit-exact against the
    oracle.  Plus the smallest case, one row of 32 columns and one token."""
    draws = synth.u64(64, 0, synth.stream_id(74))
    cases = [(1, 32, 1, (2, 4))]
    for k in range(12):
        d = [int(x) for x in draws[4 * k: 4 * k + 4]]
        rows = 1 + d[0] % 700
        cols = 32 * (1 + d[1] % 100)
        T = 1 + d[2] % 700
        if rows * cols * T > 120_000_000:  # keep the oracle to seconds
            T = max(1, 120_000_000 // (rows * cols))
        cases.append((rows, cols, T, PATTERNS[d[3] % 4]))
    for ci, (rows, cols, T, (N, M)) in enumerate(cases):
        W, X = gen(rows, cols, T, 100 + ci, exact=True)
        ov, om, v, m = dev_packed(orc, W, N, M)
        y_ref, _ = oracle_Y(orc, ov, om, cols, X)
        want = orc.round_f16(y_ref).reshape(y_ref.shape)
        Xd = to_dev(X)
        for variant in range(nm.nm_spmm_prefill_variant_count()):
            for splits in (1, 2 + (ci + variant) % 9):
                got = from_dev(nm.nm_spmm_prefill(v, m, Xd, variant=variant, splits=splits))
                bad = np.argwhere(got != want)
                assert bad.size == 0, (f"rows {rows} cols {cols} T {T} {N}:{M} variant {variant} "
                                       f"splits {splits}: {len(bad)} mismatches, first "
                                       f"{bad[:3].tolist()}")
    assert nm.nm_wait_timeouts() == 0

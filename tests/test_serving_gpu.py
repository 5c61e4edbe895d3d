"""Serving-path behaviour of the library on the GPU: CUDA-graph capture and
replay, concurrent streams, and non-finite activations.

Pruned weights are structural zeros: the kernels never multiply them, so
y[r] = sum over the columns c that row r KEEPS of w[r, c] * x[c].  A non-finite
x[c] therefore reaches exactly the rows that keep column c; every other row
stays finite and equal (within tolerance) to the oracle's value with that x[c]
set to zero.  Expected values come from the oracle only.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from gpu_util import f16_to_f64, from_dev, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

F16_INF = np.uint16(0x7C00)
F16_NINF = np.uint16(0xFC00)
F16_NAN = np.uint16(0x7E00)


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


def bits(t):
    return t.view(torch.int16)


def test_graph_replay_equals_eager(nm):
    """A chain of projections (SpMV, SpMV, dense GEMV, SpMV; each one's output
    the next one's input; programmatic dependent launch with early weight
    loads) captured once into a CUDA graph and replayed on fresh activations
    gives, bit for bit, what the same calls give eagerly."""
    n = 4096
    mats = [nm.nm_pack(to_dev(synth.weights(n, n, 0, synth.stream_id(60, i))), 2, 4)
            for i in range(3)]
    Wd = to_dev(synth.weights(n, n, 0, synth.stream_id(61)))
    x_static = torch.empty(n, dtype=torch.float16, device="cuda")
    bufs = [torch.empty(n, dtype=torch.float16, device="cuda") for _ in range(4)]

    def chain(x):
        nm.nm_spmv(*mats[0], x, y=bufs[0], flags=3)
        nm.nm_spmv(*mats[1], bufs[0], y=bufs[1], flags=3)
        nm.dense_gemv(Wd, bufs[1], y=bufs[2], flags=3)
        nm.nm_spmv(*mats[2], bufs[2], y=bufs[3], flags=3)
        return bufs[3]

    xs = [to_dev(synth.activations(n, 0, synth.stream_id(62, k))) for k in range(3)]
    eager = []
    for x in xs:
        eager.append(chain(x).clone())
    assert all(bool(torch.isfinite(e.float()).all()) for e in eager)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):          # warm the calls on the capture stream
        x_static.copy_(xs[0])
        chain(x_static)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain(x_static)
    for x, e in zip(xs, eager):
        x_static.copy_(x)
        bufs[3].zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(bits(bufs[3]), bits(e))


def test_graph_replay_long_rows_and_spmm(nm):
    """The workspace paths inside a graph: rows longer than one block's x tile
    (column-sliced nm_spmv) and a batch-4 nm_spmm, each against its eager
    result."""
    rows, cols = 96, nm.nm_spmv_max_cols() + 4096
    W = synth.weights(rows, cols, 0, synth.stream_id(63, 0))
    v, m = nm.nm_pack(to_dev(W), 2, 4)
    x = to_dev(synth.activations(cols, 0, synth.stream_id(63, 1)))
    ws = torch.empty(max(1, nm.nm_spmv_workspace_bytes(rows, cols)), dtype=torch.uint8,
                     device="cuda")
    y = torch.empty(rows, dtype=torch.float16, device="cuda")
    r2, c2, b2 = 3000, 8192, 4
    W2 = synth.weights(r2, c2, 0, synth.stream_id(63, 2))
    v2, m2 = nm.nm_pack(to_dev(W2), 4, 8)
    X2 = to_dev(synth.normal_f16((b2, c2), 0, synth.stream_id(63, 3), synth.X_SIGMA))
    ws2 = torch.empty(max(1, nm.nm_spmm_workspace_bytes(r2, c2, b2)), dtype=torch.uint8,
                      device="cuda")
    Y2 = torch.empty((b2, r2), dtype=torch.float16, device="cuda")

    def run():
        nm.nm_spmv(v, m, x, y=y, workspace=ws)
        nm.nm_spmm(v2, m2, X2, Y=Y2, workspace=ws2)

    run()
    torch.cuda.synchronize()
    y_e, Y2_e = y.clone(), Y2.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    y.zero_()
    Y2.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(bits(y), bits(y_e))
    assert torch.equal(bits(Y2), bits(Y2_e))


def test_two_streams_concurrently(nm):
    """Independent projections launched on two streams at once (each with its
    own output and workspace) give the same bits as when run alone."""
    shapes = [(8192, 4096, 2, 4), (96, nm.nm_spmv_max_cols() + 1024, 8, 16)]
    ops = []
    for k, (rows, cols, N, M) in enumerate(shapes):
        W = synth.weights(rows, cols, 0, synth.stream_id(64, k, 0))
        v, m = nm.nm_pack(to_dev(W), N, M)
        x = to_dev(synth.activations(cols, 0, synth.stream_id(64, k, 1)))
        ws = torch.empty(max(1, nm.nm_spmv_workspace_bytes(rows, cols)), dtype=torch.uint8,
                         device="cuda")
        ops.append((v, m, x, ws, rows))
    alone = [nm.nm_spmv(v, m, x, workspace=ws).clone() for v, m, x, ws, _ in ops]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in ops]
    outs = [[torch.empty(r, dtype=torch.float16, device="cuda") for _ in range(8)]
            for *_, r in ops]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for rep in range(8):
        for (v, m, x, ws, _), s, o in zip(ops, streams, outs):
            with torch.cuda.stream(s):
                nm.nm_spmv(v, m, x, y=o[rep], workspace=ws, stream=s)
    torch.cuda.synchronize()
    for a, o in zip(alone, outs):
        for t in o:
            assert torch.equal(bits(t), bits(a))


def kept_products_sum(orc, ov, om, cols, x):
    """Per row, the fp64 sum of w * x over the row's KEPT columns only: its
    class (finite, +inf, -inf, NaN) is the class the kernel must produce."""
    Wp = f16_to_f64(orc.unpack(ov, om, cols))
    rows = Wp.shape[0]
    keep = np.zeros((rows, cols), dtype=bool)
    words = cols // 32
    for w in range(words):
        bitsw = om[:, w].astype(np.uint64)
        for b in range(32):
            keep[:, 32 * w + b] = ((bitsw >> np.uint64(b)) & np.uint64(1)) == 1
    xv = f16_to_f64(x)
    with np.errstate(invalid="ignore", over="ignore"):
        prods = np.where(keep, Wp * xv[None, :], 0.0)
        return prods.sum(axis=1)


@pytest.mark.parametrize("N,M", [(2, 4), (16, 32)])
def test_nonfinite_activations_reach_only_rows_that_keep_them(nm, orc, N, M):
    rows, cols = 2048, 4096
    W = synth.weights(rows, cols, 0, synth.stream_id(65, N, 0))
    x = synth.activations(cols, 0, synth.stream_id(65, N, 1))
    x[37] = F16_INF
    x[1000] = F16_NINF
    x[2049] = F16_NAN
    ov, om = orc.prune_pack(W, N, M)
    expect = kept_products_sum(orc, ov, om, cols, x)
    # Every class must occur for the test to mean something.
    assert np.isnan(expect).any() and np.isposinf(expect).any() and np.isneginf(expect).any()
    assert np.isfinite(expect).any()
    v, m = nm.nm_pack(to_dev(W), N, M)
    xz = x.copy()
    xz[[37, 1000, 2049]] = 0
    y_ref, s = orc.spmv_f64(ov, om, cols, xz)
    fin = np.isfinite(expect)
    for variant in range(nm.nm_spmv_variant_count()):
        got = f16_to_f64(from_dev(nm.nm_spmv(v, m, to_dev(x), variant=variant)))
        assert np.array_equal(np.isnan(got), np.isnan(expect)), f"variant {variant}"
        assert np.array_equal(np.isposinf(got), np.isposinf(expect)), f"variant {variant}"
        assert np.array_equal(np.isneginf(got), np.isneginf(expect)), f"variant {variant}"
        err = np.abs(got[fin] - y_ref[fin])
        assert np.all(err <= oracle.tolerance(s[fin])), f"variant {variant}"


def test_nonfinite_token_does_not_leak_into_other_tokens(nm, orc):
    """In a batch, a non-finite activation of one token touches only that
    token's column of Y (structural zeros on the rows, no cross-token mixing
    in the padded batch slots)."""
    rows, cols, batch = 1024, 4096, 5
    W = synth.weights(rows, cols, 0, synth.stream_id(66, 0))
    X = synth.normal_f16((batch, cols), 0, synth.stream_id(66, 1), synth.X_SIGMA)
    X[2, 77] = F16_NAN
    X[2, 3000] = F16_INF
    ov, om = orc.prune_pack(W, 2, 4)
    v, m = nm.nm_pack(to_dev(W), 2, 4)
    for variant in range(nm.nm_spmm_variant_count()):
        Y = f16_to_f64(from_dev(nm.nm_spmm(v, m, to_dev(X), variant=variant)))
        for j in range(batch):
            if j == 2:
                expect = kept_products_sum(orc, ov, om, cols, X[j])
                assert np.array_equal(np.isnan(Y[j]), np.isnan(expect)), f"variant {variant}"
                assert np.array_equal(np.isposinf(Y[j]), np.isposinf(expect))
                assert np.array_equal(np.isneginf(Y[j]), np.isneginf(expect))
                continue
            y_ref, s = orc.spmv_f64(ov, om, cols, X[j])
            assert np.all(np.abs(Y[j] - y_ref) <= oracle.tolerance(s)), f"variant {variant} token {j}"

"""Every output of the full-size workloads against the oracle, in the launch
configuration the benchmark times (the library's default plans).

For each decode-layer workload and each of its N:M patterns (aimodeling.com
article, "The Kernel Is the Other Half of the Answer": 2:4, 4:8, 8:16, 16:32
on one packed format): the packed values and masks of every row are compared
bit for bit with the oracle's prune/pack, and every row of y = W x with the
oracle's double-precision SpMV of the oracle's own packing, within
|y - y_ref| <= 2e-3 * sum|w||x| + 1e-5.  The dense GEMV is checked the same
way against the oracle's dense matvec.  Then, at full size: the fused SwiGLU
gate+up projection on every (gate, up) pair, the 4-token SpMM on the gate+up,
an 8-token SpMM on the down projection (column slices) and a 6-token one on
the qkv matrix, and a 256-token prefill (K split), each on every row and
token.

The oracle runs on every host core (tests/oracle_threads.py: disjoint row
ranges, the oracle's arithmetic unchanged), which keeps a 70B-shaped layer to
seconds per pattern."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import oracle_threads as ot
import synth
from gpu_util import WORKLOADS, f16_to_f64, from_dev, to_dev

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


def assert_every_row(y_gpu, y_ref, s, what):
    err = np.abs(f16_to_f64(y_gpu) - y_ref)
    tol = oracle.tolerance(s)
    bad = np.nonzero(~(err <= tol))
    assert bad[0].size == 0, (f"{what}: {bad[0].size} outputs out of tolerance, first at "
                              f"{[b[:4] for b in bad]}, err {err[bad][:4]}, tol {tol[bad][:4]}")


@pytest.mark.parametrize("workload", list(WORKLOADS))
def test_every_row_of_every_workload(nm, orc, workload):
    spec = WORKLOADS[workload]
    for mi, (name, (rows, cols)) in enumerate(spec["mats"].items()):
        # the benchmark's weights and activations for this matrix
        W = synth.weights(rows, cols, 0, synth.stream_id(2, mi, 0))
        x = synth.activations(cols, 0, synth.stream_id(2, mi, 1))
        Wd, xd = to_dev(W), to_dev(x)
        for N, M in spec["patterns"]:
            v, m = nm.nm_pack(Wd, N, M)
            y = from_dev(nm.nm_spmv(v, m, xd))
            gv, gm = from_dev(v), from_dev(m)
            del v, m
            ov, om = ot.prune_pack(orc, W, N, M)
            assert np.array_equal(gm, om), f"{workload}/{name} {N}:{M} masks"
            assert np.array_equal(gv, ov), f"{workload}/{name} {N}:{M} values"
            assert gv.nbytes == rows * cols and gm.nbytes == rows * cols // 8
            y_ref, s = ot.spmv(orc, ov, om, cols, x)
            assert_every_row(y, y_ref, s, f"{workload}/{name} {N}:{M}")
            del gv, gm, ov, om
        yd = from_dev(nm.dense_gemv(Wd, xd))
        yd_ref, sd = ot.matvec(orc, W, x)
        assert_every_row(yd, yd_ref, sd, f"{workload}/{name} dense")
        del Wd, xd
        torch.cuda.empty_cache()


def test_every_pair_of_the_70b_swiglu_gate_up(nm, orc):
    """h = silu(W_gate x) * (W_up x) on the 57344x8192 gate+up matrix (rows
    interleaved gate, up), every one of the 28672 outputs; the tolerance
    propagates the SpMV bound through silu and the product."""
    rows, cols = 57344, 8192
    W = synth.weights(rows, cols, 0, synth.stream_id(54, rows))
    x = synth.activations(cols, 0, synth.stream_id(55, rows))
    v, m = nm.nm_pack(to_dev(W), 2, 4)
    got = f16_to_f64(from_dev(nm.nm_spmv_swiglu(v, m, to_dev(x))))
    del v, m
    ov, om = ot.prune_pack(orc, W, 2, 4)
    y, s = ot.spmv(orc, ov, om, cols, x)
    g, u, sg, su = y[0::2], y[1::2], s[0::2], s[1::2]
    h = orc.silu_mul_f64(g, u)
    silu_g = orc.silu_mul_f64(g, np.ones_like(g))
    eg, eu = 2e-3 * sg, 2e-3 * su
    tol = 1.1 * eg * (np.abs(u) + eu) + np.abs(silu_g) * eu + 1e-3 * np.abs(h) + 1e-5
    err = np.abs(got - h)
    bad = np.nonzero(~(err <= tol))[0]
    assert bad.size == 0, f"{bad.size} pairs out of tolerance, first {bad[:4]}"
    torch.cuda.empty_cache()


def test_every_row_of_a_4_token_spmm_on_the_70b_gate_up(nm, orc):
    rows, cols, batch = 57344, 8192, 4
    W = synth.weights(rows, cols, 0, synth.stream_id(41, rows, cols))
    X = synth.normal_f16((batch, cols), 0, synth.stream_id(42, rows, cols), synth.X_SIGMA)
    v, m = nm.nm_pack(to_dev(W), 8, 16)
    Y = from_dev(nm.nm_spmm(v, m, to_dev(X)))
    del v, m
    ov, om = ot.prune_pack(orc, W, 8, 16)
    for j in range(batch):
        y_ref, s = ot.spmv(orc, ov, om, cols, X[j])
        assert_every_row(Y[j], y_ref, s, f"spmm token {j}")
    torch.cuda.empty_cache()


@pytest.mark.parametrize("rows,cols,batch", [(8192, 28672, 8), (10240, 8192, 6)])
def test_every_output_of_a_small_batch_spmm_at_full_size(nm, orc, rows, cols, batch):
    """The library's plans at full size: the 70B down projection at 8 tokens
    (column slices, partial sums through the workspace and the ordered
    combine) and the qkv matrix at 6 tokens (12-byte x slots); every row and
    token against the oracle."""
    W = synth.weights(rows, cols, 0, synth.stream_id(43, rows, cols))
    X = synth.normal_f16((batch, cols), 0, synth.stream_id(44, rows, cols), synth.X_SIGMA)
    v, m = nm.nm_pack(to_dev(W), 4, 8)
    Y = from_dev(nm.nm_spmm(v, m, to_dev(X)))
    del v, m
    ov, om = ot.prune_pack(orc, W, 4, 8)
    for j in range(batch):
        y_ref, s = ot.spmv(orc, ov, om, cols, X[j])
        assert_every_row(Y[j], y_ref, s, f"{rows}x{cols} spmm token {j} of {batch}")
    torch.cuda.empty_cache()


def test_every_output_of_a_256_token_prefill_on_the_70b_qkv(nm, orc):
    """10240x8192 at 256 tokens: the library's plan cuts K (the combine adds
    the slices' fp32 sums in order); all 256 x 10240 outputs are checked."""
    rows, cols, T = 10240, 8192, 256
    _, slices, _ = nm.nm_spmm_prefill_plan(rows, cols, T)
    W = synth.weights(rows, cols, 0, synth.stream_id(74, rows, cols, 0))
    X = synth.normal_f16((T, cols), 0, synth.stream_id(74, rows, cols, 1), synth.X_SIGMA)
    v, m = nm.nm_pack(to_dev(W), 2, 4)
    Y = nm.nm_spmm_prefill(v, m, to_dev(X))
    torch.cuda.synchronize()
    assert nm.nm_wait_timeouts() == 0
    Yh = from_dev(Y)
    del v, m, Y
    ov, om = ot.prune_pack(orc, W, 2, 4)
    Y_ref, S = ot.spmv_tokens(orc, ov, om, cols, X)
    assert_every_row(Yh, Y_ref, S, f"prefill {T} tokens, {slices} K slices")
    torch.cuda.empty_cache()

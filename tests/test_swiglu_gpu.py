"""GPU parity of the fused gate+up SwiGLU projection h = silu(W_gate x) * (W_up x)
against the oracle: the oracle's packed SpMV of the even (gate) and odd (up)
rows, then its silu_mul in double.

Tolerance, from the arithmetic: the kernel's fp32 sums g~, u~ differ from the
exact g, u by at most eps_g = 2e-3 * s_g and eps_u = 2e-3 * s_u (the SpMV
bound, s = sum |w||x|); |silu'| <= 1.1, so
  |silu(g~) u~ - silu(g) u| <= 1.1 eps_g (|u| + eps_u) + |silu(g)| eps_u,
plus the fp32 evaluation of silu and the product and the single fp16 rounding
of h (< 1e-3 |h|), plus 1e-5 absolute."""
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
    return m


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


def reference(orc, ov, om, cols, x, pair_ids=None):
    rows = om.shape[0]
    pairs = np.arange(rows // 2) if pair_ids is None else np.asarray(pair_ids)
    g, sg = orc.spmv_rows_f64(ov, om, cols, x, 2 * pairs)
    u, su = orc.spmv_rows_f64(ov, om, cols, x, 2 * pairs + 1)
    h = orc.silu_mul_f64(g, u)
    silu_g = orc.silu_mul_f64(g, np.ones_like(g))
    eg, eu = 2e-3 * sg, 2e-3 * su
    tol = 1.1 * eg * (np.abs(u) + eu) + np.abs(silu_g) * eu + 1e-3 * np.abs(h) + 1e-5
    return h, tol


def check(got, h, tol, what):
    err = np.abs(f16_to_f64(got) - h)
    bad = np.nonzero(~(err <= tol))[0]
    assert bad.size == 0, f"{what}: {bad.size} bad, first {bad[:4]} err {err[bad[:4]]} tol {tol[bad[:4]]}"


@pytest.mark.parametrize("rows,cols", [(2, 32), (66, 1056), (600, 4096), (258, 14336), (130, 5120)])
@pytest.mark.parametrize("N,M", PATTERNS)
def test_swiglu_within_tolerance(nm, orc, rows, cols, N, M):
    W = synth.weights(rows, cols, 0, synth.stream_id(50, rows, cols))
    x = synth.activations(cols, 0, synth.stream_id(51, rows, cols))
    ov, om = orc.prune_pack(W, N, M)
    got = from_dev(nm.nm_spmv_swiglu(to_dev(ov), torch.from_numpy(om.view(np.int32)).cuda(),
                                     to_dev(x)))
    h, tol = reference(orc, ov, om, cols, x)
    check(got, h, tol, f"{rows}x{cols} {N}:{M}")


@pytest.mark.parametrize("rows,cols", [(66, 1056), (600, 4096)])
def test_swiglu_every_plan(nm, orc, rows, cols):
    """Small-integer inputs make g and u exact in fp32, so every plan gives the
    same h; it must also meet the tolerance."""
    W = synth.int_f16((rows, cols), 0, synth.stream_id(52, rows), -8, 8, -6)
    x = synth.int_f16((cols,), 0, synth.stream_id(53, rows), -2, 2, 0)
    ov, om = orc.prune_pack(W, 2, 4)
    v, m, xd = to_dev(ov), torch.from_numpy(om.view(np.int32)).cuda(), to_dev(x)
    h, tol = reference(orc, ov, om, cols, x)
    first = None
    for variant in range(nm.nm_spmv_variant_count()):
        for grid in (1, 3, 152, rows // 2):
            flags = (0, 1, 3)[(variant + grid) % 3]
            got = from_dev(nm.nm_spmv_swiglu(v, m, xd, variant=variant, grid=grid, flags=flags))
            check(got, h, tol, f"variant {variant} grid {grid}")
            if first is None:
                first = got
            assert np.array_equal(got, first), (variant, grid)


def test_swiglu_rejects_odd_rows(nm):
    L = nm.lib()
    v = torch.zeros((3, 16), dtype=torch.float16, device="cuda")
    m = torch.zeros((3, 1), dtype=torch.int32, device="cuda")
    x = torch.zeros(32, dtype=torch.float16, device="cuda")
    h = torch.zeros(2, dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert L.nm_spmv_swiglu(v.data_ptr(), m.data_ptr(), 3, 32, x.data_ptr(), h.data_ptr(), s) == 2
    assert L.nm_spmv_swiglu(v.data_ptr(), m.data_ptr(), 2, 32, x.data_ptr(), x.data_ptr(), s) == 7

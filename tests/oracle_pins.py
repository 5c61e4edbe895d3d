"""Pins for the CPU oracle: checks against facts fixed independently of it.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError on
a mismatch.  They are run against the real oracle (test_oracle_pins.py) and
against copies of the oracle with planted mistakes (test_oracle_mutants.py),
which must each fail at least one pin.

What fixes the expected values (never the oracle itself):
  * numpy's IEEE binary16 conversions (a library routine);
  * exact rational arithmetic (fractions.Fraction) for dot products;
  * an order-theoretic characterisation of the kept set, checked by brute
    force over all N-subsets for small M;
  * closed forms: unit-vector inputs, exact-arithmetic inputs;
  * a hand-worked golden row (tests/golden/pack_row32.json);
  * the page's format invariants (16 set bits per word, N per group, bytes).
"""
from __future__ import annotations

import functools
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
PATTERNS = [(2, 4), (4, 8), (8, 16), (16, 32)]


# --------------------------------------------------------------------------
# independent helpers (numpy / Python only)
# --------------------------------------------------------------------------
def f16_value(bits: int) -> float:
    return float(np.array([bits], dtype=np.uint16).view(np.float16)[0])


@functools.lru_cache(maxsize=None)
def magnitude_rank_key(bits: int):
    """Ordering key of the synthetic pruner expressed through values, not bit
    masks: finite and infinite entries compare by |value|; NaNs rank above
    infinity and among themselves by payload."""
    v = f16_value(bits)
    if math.isnan(v):
        return (1, bits & 0x3FF)
    return (0, abs(v))


def kept_set_is_valid(group_bits, kept, N) -> bool:
    """The kept set S is the unique set of N entries such that no entry
    outside S outranks (larger magnitude, or equal magnitude and lower
    column) an entry inside S."""
    if len(kept) != N:
        return False
    keys = [magnitude_rank_key(int(b)) for b in group_bits]
    for i in kept:
        for j in range(len(group_bits)):
            if j in kept:
                continue
            if keys[j] > keys[i] or (keys[j] == keys[i] and j < i):
                return False
    return True


def brute_force_kept(group_bits, N):
    """Enumerate all N-subsets and return the one(s) passing the rule."""
    ok = [set(c) for c in itertools.combinations(range(len(group_bits)), N)
          if kept_set_is_valid(group_bits, set(c), N)]
    return ok


def mask_bits_of(word: int):
    return [b for b in range(32) if (int(word) >> b) & 1]


def popcounts(masks: np.ndarray) -> np.ndarray:
    m = np.ascontiguousarray(masks, dtype=np.uint32)
    return np.unpackbits(m.view(np.uint8).reshape(-1, 4), axis=1).sum(axis=1).reshape(m.shape)


def kept_columns(masks_row: np.ndarray):
    cols = []
    for w, word in enumerate(masks_row):
        cols += [32 * w + b for b in mask_bits_of(word)]
    return cols


def exact_dot(w_bits, x_bits):
    acc = Fraction(0)
    mag = Fraction(0)
    for a, b in zip(w_bits, x_bits):
        fa = Fraction(f16_value(int(a)))
        fb = Fraction(f16_value(int(b)))
        acc += fa * fb
        mag += abs(fa) * abs(fb)
    return acc, mag


# --------------------------------------------------------------------------
# binary16
# --------------------------------------------------------------------------
def pin_f16_to_f64_all_patterns(o):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = allbits.view(np.float16).astype(np.float64)
    got = np.array([o.f16_to_f64(int(b)) for b in allbits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint64), ref[~nan].view(np.uint64))


def f16_from_f64_cases(seed=0):
    rng_bits = synth.u64(4000, seed, synth.stream_id(90, 1))
    # log-uniform magnitudes 2^-30 .. 2^17, random signs
    e = (rng_bits % np.uint64(47 * 1000)).astype(np.float64) / 1000.0 - 30.0
    sgn = np.where((rng_bits >> np.uint64(40)) & np.uint64(1), -1.0, 1.0)
    vals = list(sgn * np.exp2(e))
    # exact midpoints between neighbouring binary16 values (ties -> even) and
    # their immediate double neighbours
    finite = np.arange(0, 0x7C00, 97, dtype=np.uint16)
    lo = finite.view(np.float16).astype(np.float64)
    hi = (finite + 1).view(np.float16).astype(np.float64)
    mids = (lo + hi) / 2.0
    for m in mids:
        vals += [m, np.nextafter(m, 0.0), np.nextafter(m, np.inf), -m]
    vals += [0.0, -0.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e10, -1e10,
             2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -26, 3 * 2.0 ** -25,
             2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, np.inf, -np.inf, 1.0, -1.0, 0.1, 1 / 3]
    return np.array(vals, dtype=np.float64)


def pin_f16_from_f64_matches_numpy(o):
    vals = f16_from_f64_cases()
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([o.f16_from_f64(float(v)) for v in vals], dtype=np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"binary16 rounding differs at {vals[bad[:5]]}: got {got[bad[:5]]}, numpy {ref[bad[:5]]}"
    # NaN -> a NaN with the same sign
    n = o.f16_from_f64(float("nan"))
    assert (n & 0x7C00) == 0x7C00 and (n & 0x3FF) != 0


# --------------------------------------------------------------------------
# prune + pack
# --------------------------------------------------------------------------
SPECIAL_F16 = [0x0000, 0x8000, 0x0001, 0x8001, 0x1419, 0x9419, 0x3800, 0xB800,
               0x3C00, 0x7C00, 0xFC00, 0x7E00, 0xFD00]


def pin_pack_2_4_exhaustive(o):
    """Every 4-tuple over a value set with +-0, subnormals, ties, +-inf and
    NaN, packed 2:4 and compared with brute-force subset enumeration."""
    groups = np.array(list(itertools.product(SPECIAL_F16, repeat=4)), dtype=np.uint16)
    pad = (-groups.shape[0]) % 8
    groups = np.concatenate([groups, groups[:pad]])
    W = groups.reshape(-1, 32)  # 8 groups per row
    values, masks = o.prune_pack(W, 2, 4)
    for r in range(W.shape[0]):
        for g in range(8):
            gb = [int(b) for b in W[r, 4 * g:4 * g + 4]]
            word = int(masks[r, (4 * g) // 32])
            kept = {b - 4 * g for b in mask_bits_of(word) if 4 * g <= b < 4 * g + 4}
            expect = brute_force_kept(gb, 2)
            assert len(expect) == 1 and kept == expect[0], (gb, kept, expect)
    # values: the kept entries in ascending column order
    for r in range(0, W.shape[0], 37):
        cols = kept_columns(masks[r])
        assert np.array_equal(values[r], W[r, cols])


def pin_pack_random_groups(o, seed=1):
    """Random rows with many ties (values from a 6-element set), all four
    patterns; small M by full enumeration, large M by the characterisation."""
    pool = np.array([0x0000, 0x8000, 0x3C00, 0xBC00, 0x4000, 0x3800], dtype=np.uint16)
    idx = synth.u64(16 * 64, seed, synth.stream_id(91, 1)) % np.uint64(len(pool))
    W = pool[idx.astype(np.int64)].reshape(16, 64)
    for N, M in PATTERNS:
        values, masks = o.prune_pack(W, N, M)
        for r in range(W.shape[0]):
            cols = kept_columns(masks[r])
            assert np.array_equal(values[r], W[r, cols])
            for g0 in range(0, 64, M):
                gb = [int(b) for b in W[r, g0:g0 + M]]
                kept = {c - g0 for c in cols if g0 <= c < g0 + M}
                if M <= 8:
                    expect = brute_force_kept(gb, N)
                    assert len(expect) == 1 and kept == expect[0]
                else:
                    assert kept_set_is_valid(gb, kept, N)


def pin_pack_golden_row(o):
    with open(os.path.join(GOLDEN, "pack_row32.json")) as f:
        g = json.load(f)
    row = np.array([int(h, 16) for h in g["row_f16"]], dtype=np.uint16).reshape(1, 32)
    for pat, exp in g["expected"].items():
        N, M = (int(t) for t in pat.split(":"))
        values, masks = o.prune_pack(row, N, M)
        assert int(masks[0, 0]) == int(exp["mask"], 16), (pat, hex(int(masks[0, 0])))
        assert [f"{int(v):04X}" for v in values[0]] == exp["values"], pat


def pin_format_invariants(o, seed=2):
    rows, cols = 24, 256
    W = synth.weights(rows, cols, seed, synth.stream_id(92, 1))
    sizes = set()
    for N, M in PATTERNS:
        values, masks = o.prune_pack(W, N, M)
        assert np.all(popcounts(masks) == 16)
        for r in range(rows):
            kept = np.zeros(cols, dtype=np.int64)
            kept[kept_columns(masks[r])] = 1
            assert np.all(kept.reshape(-1, M).sum(axis=1) == N)
        assert masks.nbytes == rows * cols // 8 and values.nbytes == rows * cols
        sizes.add((values.nbytes, masks.nbytes))
    assert len(sizes) == 1  # identical metadata and value bytes for all patterns


def pin_roundtrip(o, seed=3):
    rows, cols = 12, 160
    W = synth.weights(rows, cols, seed, synth.stream_id(93, 1))
    for N, M in PATTERNS:
        values, masks = o.prune_pack(W, N, M)
        dense = o.unpack(values, masks, cols)
        # unpack(pack(W)) == W with the unselected entries set to +0
        expect = np.zeros_like(W)
        for r in range(rows):
            cols_k = kept_columns(masks[r])
            expect[r, cols_k] = W[r, cols_k]
        assert np.array_equal(dense, expect)
        v2, m2 = o.prune_pack(dense, N, M)
        assert np.array_equal(v2, values) and np.array_equal(m2, masks)


def pin_pattern_nesting(o, seed=4):
    """A 2:4 mask is also a valid 4:8, 8:16 and 16:32 mask: re-packing a
    2:4-pruned matrix (kept entries nonzero) under the larger M reproduces the
    same values and masks."""
    rows, cols = 8, 128
    W = synth.weights(rows, cols, seed, synth.stream_id(94, 1))
    W[(W & 0x7FFF) == 0] = 0x3C00  # no kept zeros
    v24, m24 = o.prune_pack(W, 2, 4)
    pruned = o.unpack(v24, m24, cols)
    for N, M in PATTERNS[1:]:
        v, m = o.prune_pack(pruned, N, M)
        assert np.array_equal(v, v24) and np.array_equal(m, m24), (N, M)


def pin_count_bad_words(o, seed=5):
    rows, cols = 6, 96
    W = synth.weights(rows, cols, seed, synth.stream_id(95, 1))
    _, masks = o.prune_pack(W, 2, 4)
    assert o.count_bad_words(masks, cols) == 0
    bad = masks.copy()
    bad[0, 0] ^= 1           # popcount 15 or 17
    bad[3, 2] = 0xFFFFFFFF   # 32
    bad[5, 1] = 0x0000FFFF   # 16 set bits: still fine by the invariant
    assert o.count_bad_words(bad, cols) == 2


# --------------------------------------------------------------------------
# matvec
# --------------------------------------------------------------------------
def pin_matvec_exact_rational(o, seed=6):
    rows, cols = 5, 96
    W = synth.weights(rows, cols, seed, synth.stream_id(96, 1))
    x = synth.activations(cols, seed, synth.stream_id(96, 2))
    y, s = o.matvec_f64(W, x)
    u = 2.0 ** -53
    for r in range(rows):
        ye, se = exact_dot(W[r], x)
        bound = 1.01 * cols * u * float(se)
        assert abs(y[r] - float(ye)) <= bound, (r, y[r], float(ye))
        assert abs(s[r] - float(se)) <= bound


def pin_matvec_vs_numpy(o, seed=7):
    rows, cols = 33, 320
    W = synth.weights(rows, cols, seed, synth.stream_id(97, 1))
    x = synth.activations(cols, seed, synth.stream_id(97, 2))
    y, s = o.matvec_f64(W, x)
    Wd = W.view(np.float16).astype(np.float64)
    xd = x.view(np.float16).astype(np.float64)
    yn = Wd @ xd
    sn = np.abs(Wd) @ np.abs(xd)
    bound = 2.02 * cols * 2.0 ** -53 * sn
    assert np.all(np.abs(y - yn) <= bound)
    assert np.all(np.abs(s - sn) <= bound)


def pin_spmv_unit_vectors(o, seed=8):
    """x = e_j gives y = column j of the pruned matrix, exactly."""
    rows, cols = 7, 64
    W = synth.weights(rows, cols, seed, synth.stream_id(98, 1))
    for N, M in PATTERNS:
        values, masks = o.prune_pack(W, N, M)
        dense = o.unpack(values, masks, cols).view(np.float16).astype(np.float64)
        for j in (0, 1, 5, 31, 32, 63):
            x = np.zeros(cols, dtype=np.uint16)
            x[j] = 0x3C00
            y, _ = o.spmv_f64(values, masks, cols, x)
            assert np.array_equal(y, dense[:, j]), (N, M, j)


def pin_spmv_exact_arithmetic(o, seed=9):
    """w = k 2^-6 (|k| <= 8), x in {-2..2}: the double sum is exact, so y
    equals the integer sum times 2^-6, and its fp16 rounding is numpy's."""
    rows, cols = 9, 1024
    W = synth.int_f16((rows, cols), seed, synth.stream_id(99, 1), -8, 8, -6)
    x = synth.int_f16((cols,), seed, synth.stream_id(99, 2), -2, 2, 0)
    for N, M in [(2, 4), (16, 32)]:
        values, masks = o.prune_pack(W, N, M)
        y, _ = o.spmv_f64(values, masks, cols, x)
        for r in range(rows):
            cols_k = kept_columns(masks[r])
            k = W[r, cols_k].view(np.float16).astype(np.float64) * 64.0
            xi = x[cols_k].view(np.float16).astype(np.float64)
            exact = int(np.sum(k.astype(np.int64) * xi.astype(np.int64)))
            assert y[r] == exact / 64.0
        got16 = o.round_f16(y)
        assert np.array_equal(got16, y.astype(np.float16).view(np.uint16))


def pin_spmv_rows_equals_dense_path(o, seed=10):
    rows, cols = 10, 192
    W = synth.weights(rows, cols, seed, synth.stream_id(100, 1))
    x = synth.activations(cols, seed, synth.stream_id(100, 2))
    values, masks = o.prune_pack(W, 4, 8)
    ids = np.array([9, 0, 4], dtype=np.int64)
    y, s = o.spmv_rows_f64(values, masks, cols, x, ids)
    for i, r in enumerate(ids):
        cols_k = kept_columns(masks[r])
        ye, se = exact_dot(W[r, cols_k], x[cols_k])
        bound = 1.01 * cols * 2.0 ** -53 * float(se)
        assert abs(y[i] - float(ye)) <= bound and abs(s[i] - float(se)) <= bound


def pin_leading_dimension(o, seed=11):
    """A row stride ld > cols: packing / multiplying the first cols columns of
    a wider array equals doing it on the contiguous copy."""
    rows, cols, ld = 6, 64, 100
    Wide = synth.weights(rows, ld, seed, synth.stream_id(101, 1))
    x = synth.activations(cols, seed, synth.stream_id(101, 2))
    Wc = np.ascontiguousarray(Wide[:, :cols])
    v1, m1 = o.prune_pack(Wide, 4, 8, cols=cols)
    v2, m2 = o.prune_pack(Wc, 4, 8)
    assert np.array_equal(v1, v2) and np.array_equal(m1, m2)
    y1, s1 = o.matvec_f64(Wide, x, cols=cols)
    y2, s2 = o.matvec_f64(Wc, x)
    assert np.array_equal(y1, y2) and np.array_equal(s1, s2)
    # and the contiguous result is the exact dot product of row r's first cols
    ye, _ = exact_dot(Wc[2], x)
    assert abs(y2[2] - float(ye)) <= 1e-15


def pin_silu_mul_closed_forms(o):
    """silu(t) = t / (1 + e^-t): silu(0) = 0, silu(1) = e / (1 + e),
    silu(t) - silu(-t) = t (an identity of the logistic function), silu ~ t
    for large t and ~ 0 for very negative t; h is linear in u."""
    e = math.e
    g = np.array([0.0, 1.0, -1.0, 2.5, -2.5, 40.0, -40.0, 0.125])
    u = np.array([3.0, 1.0, 1.0, 1.0, 1.0, 1.0, 1.0, -2.0])
    h = o.silu_mul_f64(g, u)
    assert h[0] == 0.0
    assert abs(h[1] - e / (1 + e)) <= 1e-15 and abs(h[2] + 1 / (1 + e)) <= 1e-15
    assert abs((h[3] - h[4]) - 2.5) <= 1e-14
    assert abs(h[5] - 40.0) <= 1e-12 and abs(h[6]) <= 1e-15
    assert abs(h[7] - (-2.0) * o.silu_mul_f64([0.125], [1.0])[0]) <= 1e-16


ALL_PINS = [
    pin_f16_to_f64_all_patterns,
    pin_f16_from_f64_matches_numpy,
    pin_pack_2_4_exhaustive,
    pin_pack_random_groups,
    pin_pack_golden_row,
    pin_format_invariants,
    pin_roundtrip,
    pin_pattern_nesting,
    pin_count_bad_words,
    pin_matvec_exact_rational,
    pin_matvec_vs_numpy,
    pin_spmv_unit_vectors,
    pin_spmv_exact_arithmetic,
    pin_spmv_rows_equals_dense_path,
    pin_leading_dimension,
    pin_silu_mul_closed_forms,
]

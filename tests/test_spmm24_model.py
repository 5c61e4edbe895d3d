"""CPU model of how the 2:4 tensor-core SpMM (nm_spmm24) divides its work and
sums panels cut between warps.

Within each column slice the flattened (panel, unit) sequence -- 16 rows by
128 columns per unit -- is cut over the slice's warps at floor(F * W / T).  A
warp stores a panel it holds whole (one slice only); otherwise it writes a
partial (slot 0: its first panel, slot 1: its last) and adds its unit count to
the panel's counter, and the warp that completes the count sums every
contributor's partial, slice by slice in warp order, finding each slice's
first contributor by a closed form.  The model mirrors that index arithmetic
and checks that every unit lands in exactly one output, every written partial
is read (and so zeroed) exactly once, no slot is written twice, and each
counter completes exactly once."""
from __future__ import annotations

import itertools
import random

import pytest


def split_at(c, q, r, parts):
    return c * q + (c * r) // parts


def owner(u, F, T):
    """The kernel's closed form for the warp whose range holds unit u."""
    return ((u + 1) * T - 1) // F


def simulate(panels, units, T, slices=1, cs=None):
    """One call: `slices` column slices of cs units (the last one the rest),
    T warps per slice.  Returns (panels stored whole, panels combined)."""
    cs = units if cs is None else cs
    sizes = [min(cs, units - s * cs) for s in range(slices)]
    assert all(z > 0 for z in sizes) and sum(sizes) == units
    stored, slots, counters, combined, read = {}, {}, {}, {}, []
    last_arrivers = []
    for s, C in enumerate(sizes):
        F = panels * C
        q, r = divmod(F, T)
        for W in range(T):
            u0, u1 = split_at(W, q, r, T), split_at(W + 1, q, r, T)
            if u0 < u1:
                assert owner(u0, F, T) == W and owner(u1 - 1, F, T) == W
            n = u1 - u0
            if n <= 0:
                continue
            p_first = u0 // C
            panel, c = p_first, u0 - p_first * C
            acc = set()
            for k in range(n):
                acc.add((s, panel * C + c))
                if c + 1 == C or k + 1 == n:
                    pb, pe = panel * C, panel * C + C
                    whole = pb >= u0 and pe <= u1
                    if slices == 1 and whole:
                        assert panel not in stored
                        stored[panel] = acc
                    else:
                        # a slice's panel held whole by one warp has a slot of
                        # its own; a cut one goes to the warp's first/last slot
                        key = (("sp", s, panel) if whole else
                               (s * T + W, 0 if panel == p_first else 1))
                        assert key not in slots, "slot written twice"
                        slots[key] = (panel, acc)
                        mine = min(u1, pe) - max(u0, pb)
                        assert mine == len(acc)
                        counters[panel] = counters.get(panel, 0) + mine
                        if counters[panel] == units:
                            last_arrivers.append(panel)
                    acc = set()
                    panel, c = panel + 1, 0
                else:
                    c += 1
    # every cut panel completes exactly once; its last arriver combines it
    assert sorted(last_arrivers) == sorted(counters)
    for panel in last_arrivers:
        got = set()
        for s, C in enumerate(sizes):
            F = panels * C
            q, r = divmod(F, T)
            pb, pe = panel * C, panel * C + C
            V = owner(pb, F, T)
            v0 = split_at(V, q, r, T)
            assert v0 <= pb < split_at(V + 1, q, r, T)
            if owner(pe - 1, F, T) == V:  # held whole by one warp
                key = ("sp", s, panel)
                assert slots[key][0] == panel and not (got & slots[key][1])
                got |= slots[key][1]
                read.append(key)
                continue
            while v0 < pe:
                v1 = split_at(V + 1, q, r, T)
                if v1 > v0:
                    key = (s * T + V, 0 if v0 // C == panel else 1)
                    assert slots[key][0] == panel
                    assert not (got & slots[key][1])
                    got |= slots[key][1]
                    read.append(key)
                V, v0 = V + 1, v1
        assert panel not in combined and panel not in stored
        combined[panel] = got
    assert sorted(read, key=str) == sorted(slots, key=str), \
        "every partial is read (and zeroed) exactly once"
    outputs = {**stored, **combined}
    assert sorted(outputs) == list(range(panels))
    for p_, us in outputs.items():
        want = set()
        for s, C in enumerate(sizes):
            want |= {(s, p_ * C + c) for c in range(C)}
        assert us == want, p_
    return len(stored), len(combined)


@pytest.mark.parametrize("panels,units,T", [
    (1, 1, 1), (1, 1, 7), (1, 64, 1), (1, 64, 2432), (3, 5, 7), (640, 64, 3040),
    (3584, 64, 3040), (512, 224, 3040), (512, 64, 1824), (2, 3, 1000), (100, 1, 37),
])
def test_split_covers_every_unit_once(panels, units, T):
    simulate(panels, units, T)


@pytest.mark.parametrize("panels,units,T,slices", [
    (512, 224, 1520, 2), (320, 200, 1520, 2), (7, 9, 5, 3), (1, 3, 2, 3), (50, 10, 400, 4),
])
def test_column_slices_cover_every_unit_once(panels, units, T, slices):
    cs = -(-units // slices)
    slices = -(-units // cs)
    whole, cut = simulate(panels, units, T, slices, cs)
    assert whole == 0 and cut == panels  # every panel is summed over its slices


def test_split_random_shapes():
    rng = random.Random(24)
    for _ in range(300):
        units = rng.randint(1, 40)
        slices = rng.choice([1, 1, 2, 3])
        cs = -(-units // slices)
        slices = -(-units // cs)
        simulate(rng.randint(1, 90), units, rng.randint(1, 300), slices, cs)


def test_cut_panels_are_bounded_by_the_warp_count():
    """Unsliced, each boundary between two warps' ranges cuts at most one
    panel, so at most T - 1 panels go through the partials."""
    for rows, cols in [(57344, 8192), (10240, 8192), (8192, 8192), (28672, 4096)]:
        whole, cut = simulate((rows + 15) // 16, cols // 128, 152 * 20)
        assert cut <= 152 * 20 - 1 and whole + cut == (rows + 15) // 16, (rows, cols)


def group_selectors(nibble):
    """The kernel's byte-permute selectors, restated: the k-th set column of a
    4-column group (k < 2) takes half k of the group's value pair, other
    columns the zero operand (byte 4)."""
    sel, k = 0, 0
    for j in range(4):
        lo = hi = 4
        if (nibble >> j) & 1:
            if k < 2:
                lo, hi = 2 * k, 2 * k + 1
            k += 1
        sel |= (lo | (hi << 4)) << (16 * (j // 2) + 8 * (j % 2))
    return sel


def byte_perm(x, y, s):
    b = x.to_bytes(4, "little") + y.to_bytes(4, "little")
    out = bytes(b[(s >> (4 * i)) & 7] for i in range(4))
    return int.from_bytes(out, "little")


def test_group_expansion_matches_the_format():
    """For every 2:4 group (two of four columns kept), the two permutes of the
    group's value pair give the dense columns the format defines: the lower
    kept column holds the first value, the upper the second, the others 0."""
    v0, v1 = 0x1234, 0xABCD
    pair = v0 | (v1 << 16)
    for cols in itertools.combinations(range(4), 2):
        nibble = sum(1 << c for c in cols)
        sel = group_selectors(nibble)
        lo = byte_perm(pair, 0, sel & 0xFFFF)
        hi = byte_perm(pair, 0, sel >> 16)
        dense = [lo & 0xFFFF, lo >> 16, hi & 0xFFFF, hi >> 16]
        want = [0, 0, 0, 0]
        want[cols[0]], want[cols[1]] = v0, v1
        assert dense == want, (cols, [hex(d) for d in dense])
    for nibble in range(16):  # malformed groups still select only the pair or zero
        sel = group_selectors(nibble)
        assert all(((sel >> (4 * i)) & 0xF) in (0, 1, 2, 3, 4) for i in range(8))

"""CPU model of how the 2:4 tensor-core SpMM (nm_spmm24) divides its work and
sums panels cut between warps.

Within each column slice the flattened (panel, unit) sequence -- 16 rows by
128 columns per unit -- is cut over the slice's blocks at floor(F * b / B),
and each block's range over its warps the same way.  A warp stores a panel
it holds whole (one slice only); a panel cut between warps of a block is
summed from shared-memory partials by its first contributing warp after a
block barrier, and stored if the block holds it whole; otherwise the block's
partial (and, with column slices, any panel a block holds whole) goes to the
workspace, its unit count to the panel's counter, and the warp that completes
the count sums every partial, slice by slice in block order, finding each
slice's first block by a closed form.  The model mirrors that index
arithmetic and checks that every unit lands in exactly one output, every
partial is used exactly once, no slot is written twice, and each counter
completes exactly once."""
from __future__ import annotations

import itertools
import random

import pytest


def split_at(c, q, r, parts):
    return c * q + (c * r) // parts


def owner(u, F, parts):
    """The kernel's closed form for the part whose range holds unit u."""
    return ((u + 1) * parts - 1) // F


def simulate(panels, units, bps, NW, slices=1, cs=None):
    """One call: `slices` column slices of cs units (the last one the rest),
    bps blocks of NW warps per slice.  Returns (panels stored whole by one
    warp, panels summed from partials)."""
    cs = units if cs is None else cs
    sizes = [min(cs, units - s * cs) for s in range(slices)]
    assert all(z > 0 for z in sizes) and sum(sizes) == units
    stored, gslots, counters, completions = {}, {}, {}, []
    for s, C in enumerate(sizes):
        F = panels * C
        bq, br = divmod(F, bps)
        for b in range(bps):
            b0, b1 = split_at(b, bq, br, bps), split_at(b + 1, bq, br, bps)
            if b0 < b1:
                assert owner(b0, F, bps) == b and owner(b1 - 1, F, bps) == b
            nb = b1 - b0
            smem = {}   # (warp, slot) -> (panel, units)
            for w in range(NW):
                w0, w1 = b0 + nb * w // NW, b0 + nb * (w + 1) // NW
                if w0 >= w1:
                    continue
                pf = w0 // C
                panel, c, acc = pf, w0 - pf * C, set()
                for k in range(w1 - w0):
                    acc.add((s, panel * C + c))
                    if c + 1 == C or k + 1 == w1 - w0:
                        pb, pe = panel * C, panel * C + C
                        if pb >= w0 and pe <= w1:  # whole in the warp
                            if slices == 1:
                                assert panel not in stored
                                stored[panel] = acc
                            else:  # its own slot, counted by the warp
                                key = ("sp", s, panel)
                                assert key not in gslots
                                gslots[key] = (panel, acc)
                                counters[panel] = counters.get(panel, 0) + len(acc)
                                if counters[panel] == units:
                                    completions.append(panel)
                        else:
                            key = (w, 0 if panel == pf else 1)
                            assert key not in smem, "shared slot written twice"
                            smem[key] = (panel, acc)
                        acc, panel, c = set(), panel + 1, 0
                    else:
                        c += 1
            # block phase: each cut panel by its first contributing warp
            used = []
            for w in range(NW):
                w0, w1 = b0 + nb * w // NW, b0 + nb * (w + 1) // NW
                if w0 >= w1:
                    continue
                pf, pl = w0 // C, (w1 - 1) // C
                todo = []
                for p_ in sorted({pf, pl}):
                    pb, pe = p_ * C, p_ * C + C
                    if pb >= w0 and pe <= w1:
                        continue  # whole in the warp
                    if p_ == pf and not (pb == w0 or w0 == b0):
                        continue  # started in an earlier warp of the block
                    todo.append(p_)
                for p_ in todo:
                    pb, pe = p_ * C, p_ * C + C
                    got, v = set(), w
                    while v < NW:
                        v0, v1 = b0 + nb * v // NW, b0 + nb * (v + 1) // NW
                        if v0 >= min(pe, b1):
                            break
                        if v1 > v0:
                            key = (v, 0 if v0 // C == p_ else 1)
                            assert smem[key][0] == p_ and not (got & smem[key][1])
                            got |= smem[key][1]
                            used.append(key)
                        v += 1
                    if pb >= b0 and pe <= b1 and slices == 1:
                        assert p_ not in stored
                        stored[p_] = got
                        continue
                    if pb >= b0 and pe <= b1:
                        key = ("sp", s, p_)
                    else:
                        key = (s * bps + b, 0 if p_ == b0 // C else 1)
                    assert key not in gslots, "global slot written twice"
                    gslots[key] = (p_, got)
                    counters[p_] = counters.get(p_, 0) + len(got)
                    if counters[p_] == units:
                        completions.append(p_)
            assert sorted(used) == sorted(smem), "every shared partial is used once"
    assert sorted(completions) == sorted(counters), "each counted panel completes once"
    combined, read = {}, []
    for p_ in completions:
        got = set()
        for s, C in enumerate(sizes):
            F = panels * C
            bq, br = divmod(F, bps)
            pb, pe = p_ * C, p_ * C + C
            B = owner(pb, F, bps)
            if owner(pe - 1, F, bps) == B:
                key = ("sp", s, p_)
                assert gslots[key][0] == p_ and not (got & gslots[key][1])
                got |= gslots[key][1]
                read.append(key)
                continue
            v0 = split_at(B, bq, br, bps)
            while v0 < pe:
                v1 = split_at(B + 1, bq, br, bps)
                if v1 > v0:
                    key = (s * bps + B, 0 if v0 // C == p_ else 1)
                    assert gslots[key][0] == p_ and not (got & gslots[key][1])
                    got |= gslots[key][1]
                    read.append(key)
                B, v0 = B + 1, v1
        assert p_ not in stored and p_ not in combined
        combined[p_] = got
    assert sorted(read, key=str) == sorted(gslots, key=str), \
        "every global partial is read (and zeroed) exactly once"
    outputs = {**stored, **combined}
    assert sorted(outputs) == list(range(panels))
    for p_, us in outputs.items():
        want = set()
        for s, C in enumerate(sizes):
            want |= {(s, p_ * C + c) for c in range(C)}
        assert us == want, p_
    return len(stored), len(combined)


@pytest.mark.parametrize("panels,units,bps,NW", [
    (1, 1, 1, 1), (1, 1, 7, 3), (1, 64, 1, 20), (1, 64, 152, 20), (3, 5, 7, 2),
    (640, 64, 152, 20), (3584, 64, 152, 20), (512, 64, 152, 16), (2, 3, 1000, 4),
    (100, 1, 37, 5),
])
def test_split_covers_every_unit_once(panels, units, bps, NW):
    simulate(panels, units, bps, NW)


@pytest.mark.parametrize("panels,units,bps,NW,slices", [
    (512, 224, 38, 20, 4), (320, 200, 38, 20, 4), (7, 9, 5, 3, 3), (1, 3, 2, 2, 3),
    (50, 10, 40, 4, 4), (896, 112, 76, 16, 2),
])
def test_column_slices_cover_every_unit_once(panels, units, bps, NW, slices):
    cs = -(-units // slices)
    slices = -(-units // cs)
    whole, cut = simulate(panels, units, bps, NW, slices, cs)
    assert whole == 0 and cut == panels  # every panel is summed over its slices


def test_split_random_shapes():
    rng = random.Random(24)
    for _ in range(400):
        units = rng.randint(1, 40)
        slices = rng.choice([1, 1, 2, 3])
        cs = -(-units // slices)
        slices = -(-units // cs)
        simulate(rng.randint(1, 90), units, rng.randint(1, 40), rng.randint(1, 12), slices, cs)


def test_blocks_hold_most_panels_cut_between_warps():
    """Unsliced, a panel goes through the workspace only where a block
    boundary cuts it: at most one per boundary, whatever the shape; the rest
    are summed in shared memory or stored by one warp."""
    for rows, cols in [(57344, 8192), (10240, 8192), (8192, 8192), (28672, 4096)]:
        panels = (rows + 15) // 16
        whole, cut = simulate(panels, cols // 128, 152, 20)
        assert whole + cut == panels


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

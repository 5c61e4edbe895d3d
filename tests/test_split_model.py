"""CPU model of the row/step split used by the matrix-vector kernels.

Mirrors the index arithmetic of csrc/split.cuh (block row ranges from a
quotient/remainder split, per-warp step ranges, the per-warp record of the
rows a range touches, which warp finishes which row, and the ordered sum of
rows cut between warps) and checks, for many shapes and launch sizes, that
every (row, step) is read exactly once, every row is written exactly once,
and every load stays inside the packed arrays.  Run before the kernels ever
see a GPU; the GPU parity tests then check the kernels themselves.
"""
import itertools

import pytest


def split_at(c, n, parts):
    """split.cuh's floor(n * c / parts) as the kernels compute it: with
    n = q * parts + r, c * q + floor(c * r / parts)."""
    q, r = divmod(n, parts)
    return c * q + (c * r) // parts


def split_part(c, n, parts):
    return split_at(c, n, parts), split_at(c + 1, n, parts)


def block_rows(rows, G, c):
    return split_part(c, rows, G)


def warp_range(F, NW, w):
    return split_part(w, F, NW)


def combine(NW, rinfo, pf, pl, r0, writes):
    """combine_cut_rows: thread t sums the row its warp cuts at its end, if
    the row started inside warp t, with the following warps' first-row
    partials up to the warp that reaches the row's end."""
    for t_ in range(NW):
        first, cs, last, ce = rinfo[t_]
        if first < 0 or not ce or (last == first and cs):
            continue
        total = list(pf[t_] if last == first else pl[t_])
        for u in range(t_ + 1, NW):
            if rinfo[u][0] < 0:
                continue
            total += pf[u]
            if not (rinfo[u][3] and rinfo[u][2] == last):
                break
        writes.setdefault(r0 + last, []).append(sorted(total))


def simulate(rows, T, G, NW):
    """The general kernel's control flow (cursor over flattened steps)."""
    writes = {}
    reads = {}
    for c in range(G):
        r0, r1 = block_rows(rows, G, c)
        F = (r1 - r0) * T
        pf, pl, rinfo = {}, {}, {}
        for w in range(NW):
            sb, se = warp_range(F, NW, w)
            row0, t0 = divmod(sb, T)
            row, t = row0, t0
            acc = []
            for s in range(sb, se):
                assert (row, t) == divmod(s, T)
                reads[(r0 + row, t)] = reads.get((r0 + row, t), 0) + 1
                acc.append((r0 + row, t))
                if t == T - 1 or s == se - 1:
                    whole = t == T - 1 and (row != row0 or t0 == 0)
                    if whole:
                        writes.setdefault(r0 + row, []).append(sorted(acc))
                    elif row == row0:
                        pf[w] = acc
                    else:
                        pl[w] = acc
                    acc = []
                t += 1
                if t == T:
                    t, row = 0, row + 1
            rinfo[w] = (row0 if se > sb else -1, t0 != 0, row if t != 0 else row - 1, t != 0)
        combine(NW, rinfo, pf, pl, r0, writes)
    return reads, writes


def simulate_whole_step(rows, T, G, NW, U):
    """The whole-step kernel's control flow: full batches of U steps, then
    single steps; a row is finished when its last step is done or, cut, when
    the warp's range ends inside it."""
    writes, reads = {}, {}
    for c in range(G):
        r0, r1 = block_rows(rows, G, c)
        F = (r1 - r0) * T
        pf, pl, rinfo = {}, {}, {}
        for w in range(NW):
            sb, se = warp_range(F, NW, w)
            row0, t0 = divmod(sb, T)
            row, t = row0, t0
            acc = []
            steps = list(range(sb, sb + (se - sb) // U * U)) + list(range(sb + (se - sb) // U * U, se))

            def finish(row, acc, whole):
                if whole:
                    writes.setdefault(r0 + row, []).append(sorted(acc))
                elif row == row0:
                    pf[w] = acc
                else:
                    pl[w] = acc

            for s in steps:
                assert (row, t) == divmod(s, T)
                reads[(r0 + row, t)] = reads.get((r0 + row, t), 0) + 1
                acc.append((r0 + row, t))
                t += 1
                if t == T:
                    finish(row, acc, row != row0 or t0 == 0)
                    acc, t, row = [], 0, row + 1
            if se > sb and t != 0:
                finish(row, acc, False)
            rinfo[w] = (row0 if se > sb else -1, t0 != 0, row if t != 0 else row - 1, t != 0)
        combine(NW, rinfo, pf, pl, r0, writes)
    return reads, writes


def test_split_at_is_the_floor_formula():
    """The kernels' division-free form gives exactly floor(n * c / parts)."""
    import random
    rng = random.Random(5)
    for _ in range(20000):
        parts = rng.choice([1, 2, 3, 7, 24, 152, 304, 1000, 65535])
        n = rng.choice([rng.randrange(0, 5000), rng.randrange(0, 2**31), rng.randrange(0, 2**40)])
        c = rng.randrange(0, parts + 1)
        assert split_at(c, n, parts) == n * c // parts


SHAPES = [(1, 1), (1, 4), (3, 1), (7, 3), (33, 2), (300, 2), (257, 4), (1000, 5), (4096, 4),
          (57, 28), (5, 28)]
LAUNCH = [(1, 16), (2, 16), (7, 8), (152, 16), (152, 24), (3, 24), (1000, 8)]


@pytest.mark.parametrize("rows,T", SHAPES)
def test_every_step_read_once_every_row_written_once(rows, T):
    for G, NW in LAUNCH:
        G = min(G, rows)
        reads, writes = simulate(rows, T, G, NW)
        assert set(reads) == {(r, t) for r in range(rows) for t in range(T)}
        assert all(v == 1 for v in reads.values())
        assert sorted(writes) == list(range(rows)), (rows, T, G, NW)
        for r, parts in writes.items():
            assert len(parts) == 1
            assert parts[0] == [(r, t) for t in range(T)], (rows, T, G, NW, r)


@pytest.mark.parametrize("rows,T", SHAPES)
def test_whole_step_kernel_control_flow(rows, T):
    for (G, NW), U in itertools.product(LAUNCH, (1, 2, 3, 4)):
        G = min(G, rows)
        reads, writes = simulate_whole_step(rows, T, G, NW, U)
        assert all(v == 1 for v in reads.values()) and len(reads) == rows * T
        assert sorted(writes) == list(range(rows))
        for r, parts in writes.items():
            assert len(parts) == 1 and parts[0] == [(r, t) for t in range(T)]


@pytest.mark.parametrize("cols", [32, 96, 992, 1024, 1056, 4096, 5120, 14336, 28672])
def test_lane_words_stay_inside_the_row(cols):
    words = cols // 32
    T = (words + 31) // 32
    pitch = (words + 31) // 32 * 32
    for t, lane in itertools.product(range(T), range(32)):
        w = t * 32 + lane
        if w < words:
            assert 8 * w + 8 <= 8 * words          # 256-bit value load inside the row
        assert w < pitch                           # pad-row read inside the x tile
    # the x tile: pad row, 32 rows of pitch floats, pad row.  The upper chain
    # reads row 1 + b for bfind b in {-1..31}; the lower chain reads row
    # 1 + (31 - b) for bfind b of the reversed mask in {-1..31}.
    for b in range(-1, 32):
        for row in (1 + b, 1 + (31 - b)):
            assert 0 <= row * pitch + (words - 1) < 34 * pitch


@pytest.mark.parametrize("rows,T", [(1, 1), (7, 3), (300, 8), (57, 28), (4096, 25)])
def test_spmm_slices_cover_every_step_once(rows, T):
    """Small-batch SpMM: the grid is shared by S column slices (blocks per
    slice = grid // S, at most rows); slice s covers warp-steps
    [T*s//S, T*(s+1)//S) of every row.  Every (row, step) must be read by
    exactly one block and every (row, slice) written once."""
    for S in sorted({1, 2, 3, T}):
        if S > T:
            continue
        for grid in (1, 7, 152):
            bps = max(1, min(grid // S, rows))
            G = bps * S
            reads, writes = {}, {}
            for b in range(G):
                sl, c = divmod(b, bps)
                r0, r1 = split_part(c, rows, bps)
                ts0, ts1 = split_part(sl, T, S)
                assert ts1 - ts0 <= -(-T // S)  # the widest slice fits the planned x tile
                for r in range(r0, r1):
                    for t in range(ts0, ts1):
                        reads[(r, t)] = reads.get((r, t), 0) + 1
                    writes[(r, sl)] = writes.get((r, sl), 0) + 1
            assert len(reads) == rows * T and all(v == 1 for v in reads.values())
            assert len(writes) == rows * S and all(v == 1 for v in writes.values())


@pytest.mark.parametrize("rows,T", [(1, 1), (7, 3), (300, 8), (57, 28), (4096, 4), (33, 14)])
def test_sliced_whole_step_loads_walk_each_rows_slice(rows, T):
    """The whole-step small-batch kernel walks each warp's loads by pointer
    increments: +1 step per step and, when a row's slice is done, a jump over
    the other slices' steps.  Model that walk (steps counted from the matrix
    start, as the masks pointer moves in units of one step's 32 words) and
    check it visits exactly the (row, step) pairs of the warp's range, in
    order, for every slice split of every launch size; and that the loads
    issued ahead in batches of U never run past the range's last step."""
    for S in sorted({1, 2, 3, T}):
        if S > T:
            continue
        for grid, NW, U in [(1, 16, 2), (7, 20, 2), (152, 20, 3), (152, 16, 2), (3, 24, 1)]:
            bps = max(1, min(grid // S, rows))
            for b in range(bps * S):
                sl, c = divmod(b, bps)
                r0, r1 = split_part(c, rows, bps)
                ts0, ts1 = split_part(sl, T, S)
                Ts, skip = ts1 - ts0, T - (ts1 - ts0)
                F = (r1 - r0) * Ts
                for w in range(NW):
                    sb, se = warp_range(F, NW, w)
                    if se <= sb:
                        continue
                    row0, t0 = divmod(sb, Ts)
                    ptr, lt = (r0 + row0) * T + ts0 + t0, t0
                    seen = []
                    nfull = (se - sb) // U
                    loads = nfull * U + (se - sb - nfull * U)
                    for _ in range(loads):
                        seen.append(ptr)
                        ptr += 1
                        lt += 1
                        if lt == Ts:
                            lt, ptr = 0, ptr + skip
                    want = [(r0 + s // Ts) * T + ts0 + s % Ts for s in range(sb, se)]
                    assert seen == want, (rows, T, S, grid, NW, U, b, w)

"""CPU model of the tensor-core prefill kernel's shared-memory arithmetic.

Mirrors csrc/prefill.cu's densify step bit for bit (popc rank, the two
16-bit loads, the PTX prmt byte permutes that merge them and zero the absent
columns, the 64-byte swizzle) and checks, before the kernel ever runs on a
GPU, that:
  * each stage's 128 x 32 tile is written exactly once per element, at the
    byte the 64-byte TMA swizzle would put the same (row, column) -- so the
    densified W tile and the X tile that TMA loads share one layout, the one
    the MMA descriptor names;
  * the densified row equals the unpacked row (kept values in place, +0
    elsewhere) for every mask with 16 set bits;
  * every shared-memory read stays inside the block's allocation, even for a
    corrupt mask word;
  * the shared-memory layout of each kernel variant fits a GB300 block and
    keeps the swizzled tiles 1024-byte aligned.
"""
import math

import numpy as np
import pytest

BM, BK, ROW_BYTES = 128, 32, 64
A_BYTES, V_BYTES, M_BYTES = BM * ROW_BYTES, BM * 32, BM * 4
DENSIFY_WARPS = 16
ROWS_PER_WARP = BM // DENSIFY_WARPS
VARIANTS = [(256, 2, 4), (256, 1, 7), (128, 1, 10), (64, 1, 12), (256, 2, 5)]
DENSIFY_GROUPS = [2, 2, 4, 4, 4]   # stage-parallel densify groups per variant
MMA_SPLIT = [0, 1, 1, 1, 0]        # 1: two issuers, even / odd stages into two accumulators
SMEM_OPTIN = 232448  # bytes of dynamic shared memory a GB300 block may opt into


def prmt(a, b, sel):
    """PTX prmt.b32 default mode: byte i of the result is byte (sel_i & 7) of
    the 8-byte value b:a, or that byte's sign replicated when sel_i & 8."""
    src = [(a >> (8 * k)) & 0xFF for k in range(4)] + [(b >> (8 * k)) & 0xFF for k in range(4)]
    out = 0
    for i in range(4):
        n = (sel >> (4 * i)) & 0xF
        byte = src[n & 7]
        if n & 8:
            byte = 0xFF if byte & 0x80 else 0x00
        out |= byte << (8 * i)
    return out


# prmt selectors by q: 0 -> (0, 0), 1 -> (v0, 0), 2 -> (0, v0), 3 -> (v0, v1)
SEL_LO, SEL_HI = 0x32103232, 0x54101032


def popc(v):
    return bin(v & 0xFFFFFFFF).count("1")


MW, MT_SLOT = 4, BM * 4 * 4


def mt_slots(stages):
    return (stages + MW - 1 + MW - 1) // MW


def layout(nmma, nb, stages, mt=True):
    vi = VARIANTS.index((nmma, nb, stages))
    full_ring, afull_ring = barrier_rings(stages, DENSIFY_GROUPS[vi], MMA_SPLIT[vi])
    bn = nmma * nb
    a_off = 0
    b_off = a_off + stages * A_BYTES
    v_off = b_off + stages * bn * ROW_BYTES
    m_off = v_off + stages * V_BYTES
    bar_off = m_off + (mt_slots(stages) * MT_SLOT if mt else stages * M_BYTES)
    n_bars = full_ring + stages + afull_ring + 1 + 2 * mt_slots(stages)
    slot_off = bar_off + n_bars * 8
    return dict(BN=bn, B_OFF=b_off, V_OFF=v_off, M_OFF=m_off, BAR_OFF=bar_off,
                BYTES=slot_off + 16, SMEM=slot_off + 16 + 1024)


def tma_sw64(r, byte_in_row):
    """Byte offset TMA's 64-byte swizzle gives (row r, byte b) of a tile with
    64-byte rows: 16-byte chunk bits [4:5] XOR address bits [7:8]."""
    L = r * ROW_BYTES + byte_in_row
    return L ^ (((L >> 7) & 3) << 4)


def densify(masks_row_words, values_rows, rpw=ROWS_PER_WARP):
    """Run the kernel's densify_stage<rpw> for one stage over the warps of one
    densify group (128 / rpw warps); returns {phys byte: (u32, row, column)}
    and the list of shared-memory reads (kind, address, row, used)."""
    writes, reads = {}, []
    for dw in range(BM // rpw):
        for lane in range(32):
            h, p = lane >> 3, lane & 7
            b0 = 4 * p
            below = (1 << b0) - 1
            lane_chunk = (p >> 1) ^ (h >> 1)
            in_chunk = (p & 1) * 8
            off_even = (lane_chunk << 4) + in_chunk
            off_odd = ((lane_chunk ^ 2) << 4) + in_chunk
            for i in range(rpw // 4):
                r = dw * rpw + 4 * i + h
                m = int(masks_row_words[r])
                reads.append(("M", 4 * r, r, 1))
                c = popc(m & below)
                nib = (m >> b0) & 15
                c2 = c + popc(nib & 3)
                a0, a2 = 32 * r + 2 * c, 32 * r + 2 * c2
                q_lo, q_hi = nib & 3, nib >> 2
                reads += [("V", a0, r, int(q_lo != 0)), ("V", a0 + 2, r, int(q_lo == 3)),
                          ("V", a2, r, int(q_hi != 0)), ("V", a2 + 2, r, int(q_hi == 3))]
                lo = prmt(values_rows.get(a0, 0), values_rows.get(a0 + 2, 0),
                          prmt(SEL_LO, SEL_HI, q_lo * 0x22 + 0x10))
                hi = prmt(values_rows.get(a2, 0), values_rows.get(a2 + 2, 0),
                          prmt(SEL_LO, SEL_HI, q_hi * 0x22 + 0x10))
                phys = r * ROW_BYTES + (off_odd if i & 1 else off_even)
                for off, val, col in ((0, lo, 4 * p), (4, hi, 4 * p + 2)):
                    assert phys + off not in writes, "element written twice"
                    writes[phys + off] = (val, r, col)
    return writes, reads


def random_masks(rng, rows, N, M):
    """Valid N:M masks (16 set bits per 32-bit word) drawn group by group."""
    words = np.zeros(rows, dtype=np.uint64)
    for r in range(rows):
        w = 0
        for g in range(32 // M):
            keep = rng.choice(M, size=N, replace=False)
            for k in keep:
                w |= 1 << (g * M + int(k))
        words[r] = w
    return words


@pytest.mark.parametrize("rpw", [8, 16, 32])
@pytest.mark.parametrize("N,M", [(2, 4), (4, 8), (8, 16), (16, 32)])
def test_densify_equals_unpack_and_matches_tma_swizzle(N, M, rpw):
    rng = np.random.default_rng(N)
    masks = random_masks(rng, BM, N, M)
    vals = rng.integers(1, 0x7BFF, size=(BM, 16), dtype=np.int64)   # nonzero fp16 bit patterns
    values_rows = {}
    for r in range(BM):
        for k in range(16):
            values_rows[32 * r + 2 * k] = int(vals[r, k])
    writes, reads = densify(masks, values_rows, rpw)
    assert len(writes) == BM * 16          # every (row, column pair) exactly once
    for phys, (out, r, col) in writes.items():
        assert phys == tma_sw64(r, 2 * col)
        m = int(masks[r])
        kept = [b for b in range(32) if (m >> b) & 1]
        want = []
        for b in (col, col + 1):
            want.append(int(vals[r, kept.index(b)]) if b in kept else 0)
        assert out == want[0] | (want[1] << 16), (r, col)
    for kind, addr, r, used in reads:
        if kind == "M":
            assert addr == 4 * r
        elif used:
            assert 32 * r <= addr < 32 * r + 32        # a kept value comes from its own row
        else:
            # a load whose value is not selected may sit up to two values past
            # the row (rank 16 when every kept bit lies left of the pair, + 1)
            assert 32 * r <= addr <= 32 * r + 34


def test_corrupt_masks_read_inside_the_allocation():
    """A word with more than 16 set bits makes the rank reach 31: the reads
    run up to 64 bytes past the row, which for the last row of the last stage
    lands in the mask ring that follows the value ring -- still inside the
    block's shared memory for every variant."""
    masks = np.full(BM, 0xFFFFFFFF, dtype=np.uint64)
    _, reads = densify(masks, {})
    vmax = max(a for k, a, _, _ in reads if k == "V")
    assert vmax <= 32 * (BM - 1) + 2 * 31 + 2
    for nmma, nb, stages in VARIANTS:
        for mt in (True, False):
            L = layout(nmma, nb, stages, mt)
            last_stage_v = L["V_OFF"] + (stages - 1) * V_BYTES
            assert last_stage_v + vmax + 2 <= L["BYTES"]


def test_densify_groups_split_stages_and_read_every_mask_box():
    """Group g of DG takes stages g, g + DG, ...: every stage exactly once,
    each group in increasing order, and (DG <= MW) every group touches every
    box of MW stages -- the condition under which a warp's wait on a mask
    box's barrier always sees that box's phase."""
    for dg in set(DENSIFY_GROUPS):
        assert DENSIFY_WARPS % dg == 0 and (BM // (DENSIFY_WARPS // dg)) % 8 == 0
        words = 37
        seen = []
        for g in range(dg):
            mine = list(range(g, words, dg))
            assert mine == sorted(mine)
            seen += mine
            boxes = sorted({k // MW for k in mine})
            assert boxes == list(range(boxes[-1] + 1))  # no box skipped
        assert sorted(seen) == list(range(words))


class _Barrier:
    """An mbarrier: a phase completes when its expected arrivals are in and
    its pending transaction bytes (here: copies) have landed.  A parity wait
    passes when the current phase's parity differs from the one named -- so
    on a fresh barrier a wait for parity 1 passes at once, and a waiter that
    is a phase ahead of the barrier passes too early.  Arrivals carry the
    stage they belong to, so a phase that mixes two stages is caught."""

    def __init__(self, count):
        self.count, self.arrived, self.tx, self.completed, self.tags = count, 0, 0, 0, []

    def arrive(self, tag=None, expect=0):
        self.arrived += 1
        self.tx += expect
        if tag is not None:
            self.tags.append(tag)
        self._check()

    def land(self):
        self.tx -= 1
        self._check()

    def _check(self):
        if self.arrived == self.count and self.tx == 0:
            assert len(set(self.tags)) <= 1, f"one phase collected arrivals of stages {self.tags}"
            self.completed += 1
            self.arrived, self.tags = 0, []


def barrier_rings(stages, dg, split):
    """Lengths of the kernel's stage-barrier rings.  A parity wait is exact
    only when the waiter itself waited for the barrier's previous phase, so
    each "full" barrier serves stages of one densify group only (a ring of
    lcm(STAGES, DG) barriers, not one per shared-memory slot), and each
    "afull" barrier stages of one MMA issuer only (2 * STAGES barriers when
    two issuers split an odd number of stages)."""
    full = stages * dg // math.gcd(stages, dg)
    afull = 2 * stages if split and stages % 2 else stages
    return full, afull


def _run_block(stages, dg, split, words, rng, wpg=2, rings=True, commit_last=False):
    """Event model of one block of the prefill kernel, masks by TMA: an X
    producer and a W producer (stage kt after the MMAs of stage kt - STAGES
    released its slot), the mask producer (box b after every densify warp
    released box b - slots), DG groups of densify warps (group g takes stages
    g, g + DG, ...), one or two MMA issuers (two: even / odd
    stages), and the copies and MMAs as asynchronous events that complete in
    any order (the MMAs of one issuer in issue order).  Actors and events run
    in random order with real parity-wait semantics.  Checks: every wait
    passes only once the phase it means has completed; every reader sees the
    stage it expects in each slot (values, mask box, densified tile, token
    tile); no slot is overwritten before its last reader; the block always
    completes.  `rings`: the kernel's barrier rings; False indexes every stage
    barrier by its shared-memory slot."""
    S, MWn = stages, MW
    FB, AB = barrier_rings(stages, dg, split) if rings else (stages, stages)
    slots = mt_slots(stages)
    nbox = words // MWn
    issuers = 2 if split else 1
    bars = {}
    for st in range(S):
        bars[f"empty{st}"] = _Barrier(1)
    for b in range(FB):
        bars[f"full{b}"] = _Barrier(2)
    for b in range(AB):
        bars[f"afull{b}"] = _Barrier(wpg)
    for sl in range(slots):
        bars[f"mfull{sl}"] = _Barrier(1)
        bars[f"mfree{sl}"] = _Barrier(dg * wpg)
    bars["accum"] = _Barrier(issuers)
    xslot, vslot, mslot = [-1] * S, [-1] * S, [-1] * slots
    aslot = [[-1] * wpg for _ in range(S)]
    mma_done = [False] * words
    dens_next = {}
    events = []                      # pending copies: (kind, index)
    mma_q = [[] for _ in range(issuers)]

    def wait(bar, parity, phase):
        return ("wait", bar, parity, phase)

    def producer(kind):
        for kt in range(words):
            st, u = kt % S, kt // S
            if u > 0:
                yield wait(f"empty{st}", (u - 1) & 1, u - 1)
            bars[f"full{kt % FB}"].arrive(expect=1, tag=kt)
            events.append((kind, kt))
        for kt in range(words - 1, max(-1, words - 1 - S), -1):
            yield wait(f"full{kt % FB}", (kt // FB) & 1, kt // FB)

    def mask_producer():
        for b in range(nbox):
            sl = b % slots
            if b >= slots:
                yield wait(f"mfree{sl}", ((b // slots) - 1) & 1, (b // slots) - 1)
            bars[f"mfull{sl}"].arrive(expect=1)
            events.append(("M", b))
        for b in range(max(0, nbox - slots), nbox):
            yield wait(f"mfull{b % slots}", (b // slots) & 1, b // slots)

    def densify(g, wi):
        key = (g, wi)
        box = -1
        for kt in range(g, words, dg):
            dens_next[key] = kt
            st = kt % S
            yield wait(f"full{kt % FB}", (kt // FB) & 1, kt // FB)
            if kt // MWn != box:
                box = kt // MWn
                yield wait(f"mfull{box % slots}", (box // slots) & 1, box // slots)
            assert vslot[st] == kt, f"densify of stage {kt} read the values of stage {vslot[st]}"
            assert mslot[box % slots] == box, f"stage {kt} read mask box {mslot[box % slots]}"
            aslot[st][wi] = kt
            yield ("step",)
            bars[f"afull{kt % AB}"].arrive(tag=kt)
            if kt + dg >= MWn * (kt // MWn + 1):
                bars[f"mfree{box % slots}"].arrive(tag=box)
        dens_next[key] = words
        yield wait("accum", 0, 0)
        assert all(mma_done)

    def issuer(r):
        k0, step = (r, 2) if split else (0, 1)
        for kt in range(k0, words, step):
            yield wait(f"afull{kt % AB}", (kt // AB) & 1, kt // AB)
            mma_q[r].append(kt)
        mma_q[r].append("accum")

    actors = [producer("X"), producer("V"), mask_producer()]
    actors += [densify(g, wi) for g in range(dg) for wi in range(wpg)]
    actors += [issuer(r) for r in range(issuers)]
    pending = [next(a, None) for a in actors]

    def can_run(req):
        if req[0] == "step":
            return True
        _, bar, parity, _ = req
        return (bars[bar].completed & 1) != parity

    while True:
        moves = [("actor", i) for i, req in enumerate(pending) if req is not None and can_run(req)]
        moves += [("event", i) for i in range(len(events))]
        moves += [("mma", r) for r in range(issuers) if mma_q[r]]
        if not moves:
            assert all(req is None for req in pending) and not events, "deadlock"
            break
        kind, i = moves[rng.integers(len(moves))]
        if kind == "actor":
            req = pending[i]
            if req[0] == "wait":
                _, bar, _, phase = req
                assert bars[bar].completed > phase, (
                    f"a parity wait on {bar} passed before its phase {phase} completed")
            pending[i] = next(actors[i], None)
        elif kind == "event":
            what, idx = events.pop(i)
            if what == "M":
                sl = idx % slots
                if idx >= slots:
                    old = idx - slots
                    assert all(dens_next[k] >= MWn * (old + 1) for k in dens_next), (
                        f"mask box {idx} overwrote box {old} before its last reader")
                mslot[sl] = idx
                bars[f"mfull{sl}"].land()
            else:
                st = idx % S
                assert idx < S or mma_done[idx - S], (
                    f"stage {idx} overwrote slot {st} before the MMAs of stage {idx - S}")
                (xslot if what == "X" else vslot)[st] = idx
                bars[f"full{idx % FB}"].land()
        else:
            item = mma_q[i].pop(0)
            if item == "accum":
                bars["accum"].arrive()
                continue
            st = item % S
            assert xslot[st] == item and all(a == item for a in aslot[st]), (
                f"MMA of stage {item} read tiles of stages {xslot[st]} / {aslot[st]}")
            mma_done[item] = True
            if commit_last or item + S < words:
                bars[f"empty{st}"].arrive()
    assert all(mma_done)


@pytest.mark.parametrize("vi", range(len(VARIANTS)))
def test_barrier_protocol_under_any_completion_order(vi):
    """Every variant's barrier protocol, including the two-issuer variants and the
    densify groups whose stage ring length is not a multiple of the group
    count, stays exact under random completion orders of every copy and MMA:
    each parity wait sees the phase it means, each reader its own stage, and
    the block always completes."""
    _, _, stages = VARIANTS[vi]
    dg, split = DENSIFY_GROUPS[vi], MMA_SPLIT[vi]
    assert dg <= MW
    rng = np.random.default_rng(4321 + vi)
    for words in (MW, 2 * MW, 3 * MW, 4 * MW, 9 * MW, 16 * MW):
        for _ in range(24):
            _run_block(stages, dg, split, words, rng)


@pytest.mark.parametrize("mt", [True, False])
@pytest.mark.parametrize("nmma,nb,stages", VARIANTS)
def test_layout_fits_and_is_aligned(nmma, nb, stages, mt):
    L = layout(nmma, nb, stages, mt)
    assert L["SMEM"] <= SMEM_OPTIN
    assert 2 * L["SMEM"] > SMEM_OPTIN + 1024      # one block per SM: TMEM never contended
    assert L["B_OFF"] % 1024 == 0 and (nmma * ROW_BYTES) % 1024 == 0
    assert L["BAR_OFF"] % 8 == 0
    acc_cols = L["BN"] * (2 if MMA_SPLIT[VARIANTS.index((nmma, nb, stages))] else 1)
    tmem = 32
    while tmem < acc_cols:
        tmem *= 2
    assert tmem <= 512 and acc_cols <= tmem
    # epilogue: the quadrant's warps stride the BN columns in 32-column loads
    assert L["BN"] % 32 == 0


def test_model_variants_match_the_kernel_table():
    """The variants this model checks are the kernel's: (tokens per MMA, MMAs
    per stage, stages, densify groups, two issuers) parsed from the table in
    prefill.cu, so a change there cannot leave the model checking another
    protocol."""
    import os
    import re
    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "sparse_spmv_memory_gb300", "csrc", "prefill.cu")).read()
    table = re.search(r"kVariants\[\]\s*=\s*\{(.*?)\};", src, re.S).group(1)
    rows = [tuple(int(x) for x in t.split(",")) for t in re.findall(r"\{([^{}]*)\}", table)]
    assert [(r[0], r[1], r[2]) for r in rows] == VARIANTS
    assert [r[4] for r in rows] == DENSIFY_GROUPS
    assert [r[6] for r in rows] == MMA_SPLIT
    assert all(r[3] == 1 and r[5] == DENSIFY_WARPS for r in rows)
    # the launch switch instantiates exactly these variants, case i = row i
    cases = re.findall(r"case (\d+): return tc::launch_tc<([^>]*)>", src)
    assert [int(i) for i, _ in cases] == list(range(len(rows)))
    assert [tuple(int(x) for x in a.split(",")) for _, a in cases] == rows
    # the plan's candidates name each variant with its own tile
    cand = re.search(r"kCand\[\]\s*=\s*\{(.*?)\};", src, re.S).group(1)
    for v, tokens in re.findall(r"\{(\d+),\s*(\d+),", cand):
        assert rows[int(v)][0] * rows[int(v)][1] == int(tokens), (v, tokens)


def test_instruction_and_smem_descriptors():
    """Bit positions of the kind::f16 instruction descriptor and the 64-byte
    swizzled K-major shared-memory descriptor the kernel builds."""
    def idesc(M, N):
        return (1 << 4) | ((N >> 3) << 17) | ((M >> 4) << 24)
    d = idesc(128, 256)
    assert (d >> 4) & 3 == 1                 # f32 accumulator
    assert (d >> 7) & 7 == 0 and (d >> 10) & 7 == 0   # f16 A and B
    assert (d >> 15) & 1 == 0 and (d >> 16) & 1 == 0  # both K-major
    assert (d >> 17) & 0x3F == 256 >> 3 and (d >> 24) & 0x1F == 128 >> 4
    assert d & ((1 << 23) | (1 << 29) | 0xF) == 0      # reserved/sparsity bits clear

    def sdesc(addr):
        return ((addr >> 4) & 0x3FFF) | (1 << 16) | ((512 >> 4) << 32) | (1 << 46) | (4 << 61)
    s = sdesc(0x2C400 + 32)
    assert s & 0x3FFF == (0x2C400 + 32) >> 4
    assert (s >> 32) & 0x3FFF == 32 and (s >> 46) & 3 == 1 and s >> 61 == 4


def test_teardown_drain_waits_only_on_final_uses_of_a_slot():
    """A producer's teardown waits on the stage barriers of the last STAGES
    stages of the row.  Each is the final use of its slot, so the barrier's
    last completed phase is the one waited for (a slot reused later would
    make the parity wait see a later phase and run out)."""
    for _, _, stages in VARIANTS:
        for words in range(1, 80):
            for kt in range(words - 1, max(-1, words - 1 - stages), -1):
                assert not [k for k in range(kt + 1, words) if k % stages == kt % stages]

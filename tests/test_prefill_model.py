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
    bn = nmma * nb
    a_off = 0
    b_off = a_off + stages * A_BYTES
    v_off = b_off + stages * bn * ROW_BYTES
    m_off = v_off + stages * V_BYTES
    bar_off = m_off + (mt_slots(stages) * MT_SLOT if mt else stages * M_BYTES)
    slot_off = bar_off + (3 * stages + 1 + mt_slots(stages)) * 8
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


def _run_pipeline(stages, dg, split, words, rng, warps_per_group=2):
    """Event model of one block's barrier protocol with masks by TMA: the X/W
    producer (stage kt once the MMAs of stage kt - STAGES are done), the mask
    producer (box b once every densify warp released box b - slots), densify
    warps (group g takes stages g, g + DG, ...; each needs the stage's tiles
    and its mask box in its slot, and releases the box after its last stage
    there) and one or two MMA issuers (with the K split: even / odd stages).
    Actors move in random order.  Asserts that no slot is refilled while a
    warp still has to read the box it holds, and that the block never
    deadlocks."""
    slots = mt_slots(stages)
    nbox = words // MW
    nwarps = dg * warps_per_group
    full, mma_done = [False] * words, [False] * words
    afull, released = [0] * words, [0] * nbox
    slot_box = [-1] * slots
    xw_next, mask_next = 0, 0
    warp_next = [w // warps_per_group for w in range(nwarps)]
    issuers = 2 if split else 1
    mma_next = list(range(issuers))

    def still_needs(w, b):
        return any(k // MW == b for k in range(warp_next[w], words, dg))

    while not all(mma_done):
        moves = []
        if xw_next < words and (xw_next < stages or mma_done[xw_next - stages]):
            moves.append(("xw",))
        if mask_next < nbox and (mask_next < slots or released[mask_next - slots] == nwarps):
            moves.append(("mask",))
        for w in range(nwarps):
            kt = warp_next[w]
            if kt < words and full[kt] and slot_box[(kt // MW) % slots] == kt // MW:
                moves.append(("dens", w))
        for i in range(issuers):
            kt = mma_next[i]
            if kt < words and afull[kt] == warps_per_group:
                moves.append(("mma", i))
        assert moves, "deadlock"
        m = moves[rng.integers(len(moves))]
        if m[0] == "xw":
            full[xw_next] = True
            xw_next += 1
        elif m[0] == "mask":
            s = mask_next % slots
            if slot_box[s] >= 0:
                assert not any(still_needs(w, slot_box[s]) for w in range(nwarps))
            slot_box[s] = mask_next
            mask_next += 1
        elif m[0] == "dens":
            w = m[1]
            kt = warp_next[w]
            afull[kt] += 1
            if kt + dg >= MW * (kt // MW + 1):   # this warp's last stage in the box
                released[kt // MW] += 1
            warp_next[w] += dg
        else:
            i = m[1]
            mma_done[mma_next[i]] = True
            mma_next[i] += issuers if split else 1
    assert released == [nwarps] * nbox


@pytest.mark.parametrize("vi", range(len(VARIANTS)))
def test_mask_slots_are_not_refilled_before_their_last_reader(vi):
    """Every densify group touches every box (DG <= MW) and releases it once
    per warp; the mask producer's wait on the release barrier then keeps each
    slot until its last reader is done, whatever the order the two K-split
    issuers and the groups run in, and the pipeline always completes."""
    _, _, stages = VARIANTS[vi]
    dg, split = DENSIFY_GROUPS[vi], MMA_SPLIT[vi]
    assert dg <= MW
    rng = np.random.default_rng(1234 + vi)
    for words in (MW, 2 * MW, 4 * MW, 64, 256):
        for _ in range(6):
            _run_pipeline(stages, dg, split, words, rng)


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

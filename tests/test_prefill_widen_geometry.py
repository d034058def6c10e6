"""Host model of the E4M3 prefill's widening index arithmetic (no GPU).

The tensor-core prefill over an E4M3 cache lands a K (or V) tile as 128 key
rows x 128 one-byte codes in the second 16 KB half of its 32 KB ring slot,
128B-swizzled (16-byte chunk j of row r at position j ^ (r % 8)).  Two warps
(64 threads) widen it in place into the f16 tile the MMAs read: two 64-column
halves of 128 rows x 128 bytes, the same swizzle.  Thread ct reads, for
i = 0..15, code chunk j = (ct // 8) % 8 of row r = ct % 8 + 8 i and writes f16
chunks 2 (j % 4) and 2 (j % 4) + 1 of half j // 4.  Each softmax thread
rewrites its own Q row (two 128-byte halves) in place, visiting chunk c at
position c ^ (row % 8).

This replays that arithmetic and checks what the kernel relies on:
  * every code byte of the tile is read once, every f16 byte written once;
  * f16 column k of a row comes from code column k of the same row (so the
    widened tile is the tile the bf16 path would have loaded);
  * reads stay in the slot's code half, writes in the slot;
  * the 8 lanes of each shared-memory phase of a 16-byte access touch 8
    distinct 16-byte bank groups (no bank conflicts), for the widening reads
    and writes and for the Q rewrite.
"""
from collections import Counter

KEYS, HALF = 128, 16384                 # rows per tile; bytes of one 64-column f16 half


def code_addr(r, j):
    """Byte offset (in the slot) of code chunk j (codes 16 j .. 16 j + 15) of row r."""
    return HALF + r * 128 + ((j ^ (r % 8)) << 4)


def f16_addr(r, c, hh):
    """Byte offset of f16 chunk c (columns 64 hh + 8 c .. + 7) of row r."""
    return hh * HALF + r * 128 + ((c ^ (r % 8)) << 4)


def widen_plan():
    """Per (warp, i): the lane list of (read addr, [(write addr, columns)])."""
    plan = {}
    for ct in range(64):
        warp, lane = divmod(ct, 32)
        j, r7 = (ct >> 3) & 7, ct & 7
        c0 = 2 * (j & 3)
        for i in range(KEYS // 8):
            r = r7 + 8 * i
            rd = code_addr(r, j)
            # f16 chunk c0 holds codes 16 j .. 16 j + 7, chunk c0 + 1 the next 8
            wr = [(f16_addr(r, c0, j >> 2), (r, 16 * j)),
                  (f16_addr(r, c0 + 1, j >> 2), (r, 16 * j + 8))]
            plan.setdefault((warp, i), []).append((lane, rd, wr, r, j))
    return plan


def test_every_code_read_once_and_every_f16_chunk_written_once():
    reads, writes = Counter(), Counter()
    for accesses in widen_plan().values():
        for _, rd, wr, _, _ in accesses:
            for b in range(16):
                reads[rd + b] += 1
            for addr, _ in wr:
                for b in range(16):
                    writes[addr + b] += 1
    assert set(reads) == set(range(HALF, 2 * HALF)) and set(reads.values()) == {1}
    assert set(writes) == set(range(2 * HALF)) and set(writes.values()) == {1}


def test_widened_columns_come_from_the_same_row_and_columns():
    # physical f16 chunk -> (row, first column) must match the bf16 tile layout
    for accesses in widen_plan().values():
        for _, _, wr, r, j in accesses:
            for addr, (row, col) in wr:
                hh, rest = divmod(addr, HALF)
                prow, pos = divmod(rest, 128)
                c = (pos >> 4) ^ (prow % 8)
                assert prow == row == r
                assert 64 * hh + 8 * c == col
                # and the codes read for those columns are row r's codes 16 j ..
                assert col in (16 * j, 16 * j + 8)


def _conflict_free(addrs):
    """8 lanes of a 16-byte access: distinct 16-byte bank groups (addr / 16 % 8)."""
    groups = [(a >> 4) & 7 for a in addrs]
    return len(set(groups)) == len(groups)


def test_widening_phases_are_conflict_free():
    for accesses in widen_plan().values():
        lanes = sorted(accesses)
        assert len(lanes) == 32
        for ph in range(4):
            phase = lanes[8 * ph: 8 * ph + 8]
            assert _conflict_free([rd for _, rd, _, _, _ in phase])
            for k in range(2):
                assert _conflict_free([wr[k][0] for _, _, wr, _, _ in phase])


def test_q_rewrite_is_in_place_and_conflict_free():
    # softmax thread `row` (0..127) of a warpgroup visits chunk c of each half
    # at position (c & 7) ^ (row % 8); positions cover the row once, and the 8
    # consecutive rows of a phase hit distinct bank groups
    for row in range(KEYS):
        pos = [(c >> 3) * HALF + row * 128 + (((c & 7) ^ (row & 7)) * 16) for c in range(16)]
        assert sorted(pos) == [h * HALF + row * 128 + 16 * k for h in range(2) for k in range(8)]
    for c in range(16):
        for base in range(0, KEYS, 8):
            addrs = [(c >> 3) * HALF + row * 128 + (((c & 7) ^ (row & 7)) * 16)
                     for row in range(base, base + 8)]
            assert _conflict_free(addrs)


def test_model_catches_an_unswizzled_read():
    # reading chunk j at position j (ignoring the swizzle) puts a phase's 8
    # rows on one bank group: the check above must fail for it
    addrs = [HALF + r * 128 + (0 << 4) for r in range(8)]
    assert not _conflict_free(addrs)

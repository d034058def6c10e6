"""Host model of the fused write's coverage (pkv_write_attention_varlen).

In a decode-class step every decode CTA - one per (split s, KV head, row tile
z, request) - stores the new-token rows at positions [max(L - n, 16 b0),
key_end) of its range before reading them.  The step is only correct if every
new token of every request is stored by some CTA, and if every CTA that reads
a new-token row stores it first.  This replays the kernel's geometry (row
tiles of R rows, the causal limit of the tile's last row, contiguous equal
block ranges per split) over random shapes and checks both properties.
"""

import numpy as np
import pytest

BLOCK = 16


def rows_per_tile(group: int) -> int:
    return 4 if group <= 4 else (8 if group <= 8 else 16)


def cta_ranges(L: int, n: int, group: int, splits: int, causal: bool = True):
    """(read range, stored range) of positions for every CTA of one request
    and KV head, as the decode kernel computes them."""
    R = rows_per_tile(group)
    rows_total = group * n
    out = []
    for z in range(-(-rows_total // R)):
        rho0 = z * R
        nrows = min(R, rows_total - rho0)
        i_last = (rho0 + nrows - 1) // group
        kv_len = (L - n + i_last + 1) if causal else L
        nblk = -(-kv_len // BLOCK)
        blk_lo = 0
        for s in range(splits):
            if splits > 1:
                per = -(-(nblk - blk_lo) // splits)
                b0 = blk_lo + min(s * per, nblk - blk_lo)
                b1 = min(b0 + per, nblk)
            else:
                if s:
                    continue
                b0, b1 = blk_lo, nblk
            if b0 >= b1:
                continue
            key_end = min(kv_len, b1 * BLOCK)
            read = (b0 * BLOCK, key_end)
            stored = (max(L - n, b0 * BLOCK), key_end)
            out.append((read, stored))
    return out


@pytest.mark.parametrize("seed", range(40))
def test_every_new_token_is_stored_and_every_reader_stores_first(seed):
    rng = np.random.default_rng(seed)
    for _ in range(200):
        n = int(rng.integers(1, 5))                  # decode-class
        L = int(rng.integers(n, 3000))
        group = int(rng.choice([1, 2, 4, 8, 16]))
        splits = int(rng.choice([1, 2, 3, 7, 16, 64]))
        causal = bool(rng.integers(0, 2))
        ctas = cta_ranges(L, n, group, splits, causal)
        stored = set()
        for (r0, r1), (s0, s1) in ctas:
            stored.update(range(s0, s1))
            # a CTA reading a new-token row stores it itself
            for p in range(max(r0, L - n), r1):
                assert s0 <= p < s1, (L, n, group, splits, p)
        assert stored == set(range(L - n, L)), (L, n, group, splits, causal)

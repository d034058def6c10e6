"""Host model of the split-KV decode kernel's key ranges, with sliding windows.

For a row tile (R rows = GQA group x new tokens) the kernel starts its block
range at the block of its first row's window start, splits [blk_lo, nblk)
into contiguous equal runs of whole blocks, and each row then keeps the keys
lo_row <= j < lim_row of each run.  This replays that arithmetic and checks
that, for every row, the splits together visit each key the row may see
exactly once and nothing outside the request's context.
"""

import numpy as np
import pytest

BLOCK = 16


def rows_per_tile(group):
    return 4 if group <= 4 else (8 if group <= 8 else 16)


def tile_ranges(L, n, group, splits, window, z, causal=True):
    R = rows_per_tile(group)
    rho0 = z * R
    nrows = min(R, group * n - rho0)
    i_last = (rho0 + nrows - 1) // group
    kv_len = (L - n + i_last + 1) if causal else L
    nblk = -(-kv_len // BLOCK)
    key_lo = max(0, L - n + rho0 // group - window + 1) if window > 0 else 0
    blk_lo = min(key_lo // BLOCK, nblk)
    out = []
    for s in range(splits):
        if splits > 1:
            per = -(-(nblk - blk_lo) // splits)
            b0 = blk_lo + min(s * per, nblk - blk_lo)
            b1 = min(b0 + per, nblk)
        else:
            if s:
                continue
            b0, b1 = blk_lo, nblk
        if b0 < b1:
            out.append((b0 * BLOCK, min(kv_len, b1 * BLOCK)))
    rows = []
    for rho in range(nrows):
        i = (rho0 + rho) // group
        lim = (L - n + i + 1) if causal else L
        lo = (L - n + i - window + 1) if window > 0 else -(1 << 30)
        rows.append((max(lo, 0), lim))
    return out, rows


@pytest.mark.parametrize("seed", range(30))
def test_each_visible_key_once(seed):
    rng = np.random.default_rng(seed)
    for _ in range(150):
        n = int(rng.integers(1, 5))
        L = int(rng.integers(n, 2500))
        group = int(rng.choice([1, 2, 4, 8, 16]))
        splits = int(rng.choice([1, 2, 3, 5, 16, 64]))
        window = int(rng.choice([0, 1, 7, 16, 17, 100, 1000, 5000]))
        causal = bool(rng.integers(0, 2))
        R = rows_per_tile(group)
        for z in range(-(-group * n // R)):
            ranges, rows = tile_ranges(L, n, group, splits, window, z, causal)
            for lo, lim in rows:
                hits = np.zeros(L, dtype=int)
                for a, b in ranges:
                    assert 0 <= a < b <= L
                    hits[max(a, lo):max(min(b, lim), max(a, lo))] += 1
                want = np.zeros(L, dtype=int)
                want[lo:lim] = 1
                assert np.array_equal(hits, want), (L, n, group, splits, window, z)

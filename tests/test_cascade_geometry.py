"""Host model of the cascade's packed prefix pass (tensor-core mode).

A CTA (tile pair p, KV head g, split s) holds two 128-row tiles; row `row`
of tile t is the packed row rho = (2 p + t) * 128 + row, i.e. token
rho // group with query head g * group + rho % group, and its Q comes from a
TMA box of {64 columns, group heads, 128 / group tokens} starting at token
(2 p + t) * 128 / group.  Split s takes the prefix's 128-key tiles
[s * per, s * per + per) cut at the end.  This replays that geometry and checks
that every (token, query head) row is computed exactly once per split, that
the box rows are those rows in the same order, that the splits partition the
key tiles, and that the partials' workspace rows never collide.
"""

import numpy as np
import pytest

ROWS = 128


def packed_rows(T, group, g):
    """{(token, head): count} over every CTA row of KV head g."""
    seen = {}
    pairs = -(-T * group // (2 * ROWS))
    for p in range(pairs):
        for t in range(2):
            tok0 = (2 * p + t) * (ROWS // group)        # the Q box's first token
            for row in range(ROWS):
                rho = (2 * p + t) * ROWS + row
                tk, h = rho // group, g * group + rho % group
                # the box row `row` is token tok0 + row // group, head row % group
                assert (tok0 + row // group, g * group + row % group) == (tk, h)
                if tk < T:
                    seen[(tk, h)] = seen.get((tk, h), 0) + 1
    return seen


def split_tiles(P, splits):
    ntk = -(-P // 128)
    per = -(-ntk // splits)
    out = []
    for s in range(splits):
        base = min(s * per, ntk)
        out.append(list(range(base, base + max(0, min(per, ntk - base)))))
    return out, ntk


@pytest.mark.parametrize("group", [2, 4, 8, 16])
@pytest.mark.parametrize("T", [1, 3, 31, 32, 64, 65, 200])
def test_every_row_once(T, group):
    hkv = 2
    for g in range(hkv):
        seen = packed_rows(T, group, g)
        want = {(tk, g * group + j) for tk in range(T) for j in range(group)}
        assert set(seen) == want and all(c == 1 for c in seen.values())


@pytest.mark.parametrize("P,splits", [(16, 1), (16, 3), (128, 2), (4096, 16), (4096, 63),
                                      (1000, 7), (2048, 64)])
def test_splits_partition_the_key_tiles(P, splits):
    tiles, ntk = split_tiles(P, splits)
    flat = [k for ts in tiles for k in ts]
    assert sorted(flat) == list(range(ntk)) and len(flat) == ntk


def test_partial_rows_do_not_collide():
    rng = np.random.default_rng(3)
    for _ in range(50):
        T = int(rng.integers(1, 300))
        hkv = int(rng.integers(1, 5))
        group = int(rng.choice([2, 4, 8]))
        S = int(rng.integers(1, 17))
        hq = hkv * group
        rows = set()
        for s in range(S + 1):                        # S prefix splits + the own-key slot
            for tk in range(T):
                for h in range(hq):
                    w = (s * T + tk) * hq + h
                    assert w not in rows
                    rows.add(w)
        assert len(rows) == (S + 1) * T * hq

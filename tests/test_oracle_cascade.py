"""Pins of the shared-prefix oracle (oracle/cascade.py).

The plain result (attention over shared ++ own blocks) is checked against the
brute-force masked-matrix formulation; the two-level form a cascade kernel
computes (prefix partial over all rows, suffix partial per request, LSE merge)
must equal it to float64 rounding; q = 0 gives the mean of every visible
value, prefix and suffix alike.
"""

import math

import numpy as np
import pytest

import workloads
from oracle import brute, cascade, flatten


def _parts(w):
    P = w.shared_blocks * 16
    meta = flatten.flatten(w.requests)
    shared = w.requests[0].blocks[:w.shared_blocks]
    suffix_table = [r.blocks[w.shared_blocks:] for r in w.requests]
    suffix_lens = [r.computed + r.scheduled - P for r in w.requests]
    return meta, shared, suffix_table, suffix_lens


def _cascade_workload(seed, shared_blocks, shape, hq=4, hkv=2, d=16):
    return workloads.build_cascade("c", "f32", hq, hkv, d, shared_blocks, shape, seed=seed)


SHAPES = [[(0, 1), (5, 1), (30, 2), (17, 4), (3, 3)], [(40, 7), (0, 1)], [(0, 1)] * 6]


@pytest.mark.parametrize("shared_blocks", [0, 1, 3])
@pytest.mark.parametrize("shape", SHAPES)
def test_cascade_matches_brute_force(shared_blocks, shape):
    w = _cascade_workload(3 + shared_blocks, shared_blocks, shape)
    meta, shared, suffix_table, suffix_lens = _parts(w)
    kw = dict(num_q_heads=4, num_kv_heads=2, softmax_scale=w.softmax_scale, dtype="f32")
    o, _ = cascade.attention(w.q, w.k_pool, w.v_pool, meta["query_start_loc"], suffix_lens,
                             suffix_table, shared, **kw)
    table, lens = cascade.full_tables(shared, suffix_table, suffix_lens)
    b = brute.attention(w.q, w.k_pool, w.v_pool, meta["query_start_loc"], lens, table, **kw)
    assert np.abs(o - b).max() < 1e-12


@pytest.mark.parametrize("shared_blocks", [0, 1, 4])
@pytest.mark.parametrize("shape", SHAPES)
def test_two_level_merge_equals_plain_attention(shared_blocks, shape):
    w = _cascade_workload(9 + shared_blocks, shared_blocks, shape)
    meta, shared, suffix_table, suffix_lens = _parts(w)
    kw = dict(num_q_heads=4, num_kv_heads=2, softmax_scale=w.softmax_scale, dtype="f32")
    args = (w.q, w.k_pool, w.v_pool, meta["query_start_loc"], suffix_lens, suffix_table, shared)
    o, lse = cascade.attention(*args, **kw)
    o2, lse2 = cascade.two_level(*args, **kw)
    assert np.abs(o - o2).max() < 1e-12 and np.abs(lse - lse2).max() < 1e-12


def test_zero_query_averages_prefix_and_suffix_values():
    w = _cascade_workload(21, 2, [(10, 2), (0, 1)], hq=2, hkv=1, d=8)
    w.q[:] = 0.0
    meta, shared, suffix_table, suffix_lens = _parts(w)
    o, lse = cascade.attention(w.q, w.k_pool, w.v_pool, meta["query_start_loc"], suffix_lens,
                               suffix_table, shared, num_q_heads=2, num_kv_heads=1,
                               softmax_scale=0.5, dtype="f32")
    flat = w.v_pool.reshape(-1, 1, 8).astype(np.float64)
    t = 0
    for r in w.requests:
        L, n = r.computed + r.scheduled, r.scheduled
        slots = [b * 16 + j for b in r.blocks for j in range(16)][:L]
        for i in range(n):
            vis = L - n + i + 1
            assert np.allclose(o[t, 0], flat[slots[:vis], 0].mean(axis=0), atol=1e-13, rtol=0)
            assert abs(lse[t, 0] - math.log(vis)) < 1e-13
            t += 1


def test_planted_causal_prefix_pass_is_caught(monkeypatch):
    # a cascade that masked the prefix causally (as if each row sat inside it)
    # must disagree with the plain result
    from oracle import ref
    w = _cascade_workload(13, 3, [(4, 1), (0, 2)])
    meta, shared, suffix_table, suffix_lens = _parts(w)
    kw = dict(num_q_heads=4, num_kv_heads=2, softmax_scale=w.softmax_scale, dtype="f32")
    args = (w.q, w.k_pool, w.v_pool, meta["query_start_loc"], suffix_lens, suffix_table, shared)
    o, _ = cascade.attention(*args, **kw)
    orig = ref.attention
    monkeypatch.setattr(ref, "attention",
                        lambda *a, causal=True, **k: orig(*a, causal=True, **k))
    o2, _ = cascade.two_level(*args, **kw)
    assert np.abs(o - o2).max() > 1e-6

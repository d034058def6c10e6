"""Online softmax, split-KV partials and their log-sum-exp merge, in float64.

Follows "Inside the engine: kernels, CUDA graphs and the life of a request":

* section "Never materialise the TxT matrix": keys and values stream past the
  query tile by tile; a running maximum m and running denominator l are kept,
  and whenever the maximum moves the accumulator (and l) is rescaled by
  e^(m_old - m_new).  The result equals the full softmax, and m only rises.
* section "Prefill has a full grid; decode at batch 1 has almost none": the
  key axis is split, each split runs the same online softmax over its part,
  and a second reduction combines the partials without changing the result.

The page states no combine formula; the reading taken is the standard exact
one: each split s reports o_s = acc_s / l_s and lse_s = m_s + ln l_s (an empty
split reports lse = -inf), and the merge is
M = max_s lse_s, w_s = e^(lse_s - M), o = sum_s w_s o_s / sum_s w_s.
The split partition is contiguous, equal-size runs of 16-token blocks (the page
says any split leaves the result unchanged).
"""

from __future__ import annotations

import math

import numpy as np


def online_softmax(s: np.ndarray, v: np.ndarray, tile: int):
    """Online softmax of one row: scores ``s`` [L], values ``v`` [L, D].

    Returns (o, lse, m_trace) where m_trace is the running maximum after each
    tile.  An empty row gives o = 0, lse = -inf.
    """
    m, l = -math.inf, 0.0
    acc = np.zeros(v.shape[1])
    trace = []
    for t0 in range(0, s.shape[0], tile):
        st, vt = s[t0:t0 + tile], v[t0:t0 + tile]
        m_new = max(m, float(st.max()))
        alpha = math.exp(m - m_new) if m != -math.inf else 0.0
        p = np.exp(st - m_new)
        acc = acc * alpha + p @ vt
        l = l * alpha + float(p.sum())
        m = m_new
        trace.append(m)
    if l == 0.0:
        return np.zeros(v.shape[1]), -math.inf, trace
    return acc / l, m + math.log(l), trace


def split_ranges(num_keys: int, num_splits: int, block_size: int = 16):
    """Contiguous key ranges of ``num_splits`` equal runs of whole blocks."""
    nblocks = -(-num_keys // block_size)
    per = -(-nblocks // num_splits) if nblocks else 0
    out = []
    for s in range(num_splits):
        a = min(s * per * block_size, num_keys)
        b = min((s + 1) * per * block_size, num_keys)
        out.append((a, b))
    return out


def combine(partials):
    """Merge split partials [(o_s, lse_s), ...] by their log-sum-exp weights."""
    lses = np.array([lse for _, lse in partials], dtype=np.float64)
    M = lses.max()
    if M == -math.inf:
        return np.zeros_like(partials[0][0]), -math.inf
    w = np.exp(lses - M)
    o = sum(wi * oi for wi, (oi, _) in zip(w, partials)) / w.sum()
    return o, M + math.log(w.sum())


def split_attention_row(s: np.ndarray, v: np.ndarray, num_splits: int, tile: int = 16,
                        block_size: int = 16):
    """One row of attention the split-KV way: online softmax per split, then merge."""
    parts = []
    for a, b in split_ranges(s.shape[0], num_splits, block_size):
        if b > a:
            o, lse, _ = online_softmax(s[a:b], v[a:b], tile)
        else:
            o, lse = np.zeros(v.shape[1]), -math.inf
        parts.append((o, lse))
    return combine(parts)

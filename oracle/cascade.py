"""Shared-prefix (cascade) attention in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

"Anatomy of a serving engine", section "Capacity belongs to the KV cache
manager": PagedAttention lets requests share blocks for a common prefix; "Inside the engine ...",
section "Attention over a block table, not a contiguous tensor": a request's
keys are whatever blocks its table names.  The reading taken for a shared
prefix: every request in the batch starts with the same ``shared_table``
blocks (P = 16 * len(shared_table) keys), followed by its own
``suffix_lens[r]`` keys in ``suffix_table[r]``; its context is L = P +
suffix_lens[r] and its n new tokens are the last n of those (all inside its
own suffix).  The result is plain paged attention with the table
shared_table ++ suffix_table[r] - which is what ``attention`` computes.

``two_level`` takes the decomposition a cascade kernel uses instead: each row's
attention over the prefix alone (every prefix key is visible to every new row,
which sits after the prefix), its attention over its own suffix alone
(causal), and the log-sum-exp merge of the two partials ("Prefill has a full
grid ...": a split of the key axis changes nothing about the result).  The
pins check that it equals ``attention``.
"""

from __future__ import annotations

import numpy as np

from . import merge, ref


def full_tables(shared_table, suffix_table, suffix_lens, block_size: int = 16):
    """Per-request tables shared ++ own, and the full context lengths."""
    shared = [int(b) for b in shared_table]
    P = len(shared) * block_size
    nb_max = len(shared) + max((len(row) for row in suffix_table), default=0)
    table = np.zeros((len(suffix_lens), max(nb_max, 1)), dtype=np.int32)
    for r, row in enumerate(suffix_table):
        blocks = shared + [int(b) for b in row]
        table[r, :len(blocks)] = blocks
    lens = np.asarray(suffix_lens, dtype=np.int64) + P
    return table, lens


def attention(q, k_cache, v_cache, query_start_loc, suffix_lens, suffix_table, shared_table, *,
              num_q_heads, num_kv_heads, softmax_scale, dtype="f32", block_size=16,
              tokens=None):
    """(o, lse) of the batch: plain paged attention over shared ++ own blocks."""
    table, lens = full_tables(shared_table, suffix_table, suffix_lens, block_size)
    return ref.attention(q, k_cache, v_cache, query_start_loc, lens, table,
                         num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                         softmax_scale=softmax_scale, causal=True, block_size=block_size,
                         dtype=dtype, tokens=tokens)


def two_level(q, k_cache, v_cache, query_start_loc, suffix_lens, suffix_table, shared_table, *,
              num_q_heads, num_kv_heads, softmax_scale, dtype="f32", block_size=16):
    """The same result as prefix partial + suffix partial merged by LSE."""
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    n_tok = int(qsl[-1])
    P = len(shared_table) * block_size
    # prefix partial: all rows of the batch as one request over the P shared
    # keys, no mask (every new row sits after the prefix)
    o1, lse1 = ref.attention(q[:n_tok], k_cache, v_cache, np.array([0, n_tok]), np.array([P]),
                             np.asarray([list(shared_table) or [0]], dtype=np.int64),
                             num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                             softmax_scale=softmax_scale, causal=False, block_size=block_size,
                             dtype=dtype)
    if P == 0:
        o1 = np.zeros_like(o1)
        lse1 = np.full_like(lse1, -np.inf)
    # suffix partial: each request over its own keys, causal
    width = max(max((len(r) for r in suffix_table), default=0), 1)
    table = np.zeros((len(suffix_lens), width), dtype=np.int64)
    for r, row in enumerate(suffix_table):
        table[r, :len(row)] = row
    o2, lse2 = ref.attention(q, k_cache, v_cache, qsl, np.asarray(suffix_lens), table,
                             num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                             softmax_scale=softmax_scale, causal=True, block_size=block_size,
                             dtype=dtype)
    o = np.empty_like(o2)
    lse = np.empty_like(lse2)
    for t in range(n_tok):
        for h in range(num_q_heads):
            o[t, h], lse[t, h] = merge.combine([(o1[t, h], lse1[t, h]), (o2[t, h], lse2[t, h])])
    return o, lse

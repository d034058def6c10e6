"""Flat-batch metadata and the slot-mapped KV write (oracle side).

Follows "Model execution", section "Flattening a step" (the tensor table) and
its ``flatten_batch.py`` worked example: every scheduled token of every
request is concatenated into one flat batch; ``query_start_loc`` holds the
cumulative offsets of each request's tokens, ``seq_lens`` each request's total
context after this step, ``block_table`` the physical blocks of its context and
``slot_mapping`` the physical slot of each new token,
``block_id * block_size + offset``.  Blocks hold 16 tokens ("Inside the
engine ...", section "Attention over a block table, not a contiguous tensor").
"""

from __future__ import annotations

import numpy as np


def flatten(requests, block_size: int = 16) -> dict:
    """Build the flat-batch tensors of one step from its schedule.

    ``requests``: sequence of objects with ``computed`` (tokens already in
    the cache), ``scheduled`` (tokens computed this step) and ``blocks`` (the
    request's block table, logical order).
    """
    positions, slots, req_index = [], [], []
    for r, req in enumerate(requests):
        for pos in range(req.computed, req.computed + req.scheduled):
            logical_block, offset = divmod(pos, block_size)
            positions.append(pos)
            slots.append(req.blocks[logical_block] * block_size + offset)
            req_index.append(r)
    qsl = [0]
    for req in requests:
        qsl.append(qsl[-1] + req.scheduled)
    seq_lens = [req.computed + req.scheduled for req in requests]
    width = max([len(req.blocks) for req in requests] + [1])
    table = np.zeros((len(requests), width), dtype=np.int64)
    for r, req in enumerate(requests):
        table[r, :len(req.blocks)] = req.blocks
    return {
        "positions": np.array(positions, dtype=np.int64),
        "slot_mapping": np.array(slots, dtype=np.int64),
        "request_index": np.array(req_index, dtype=np.int64),
        "query_start_loc": np.array(qsl, dtype=np.int64),
        "seq_lens": np.array(seq_lens, dtype=np.int64),
        "block_table": table,
        "logits_indices": np.array([q - 1 for q in qsl[1:]], dtype=np.int64),
    }


def context_slots(req, block_size: int = 16) -> np.ndarray:
    """Physical slot of every logical position 0..seq_len-1 of one request."""
    out = []
    for pos in range(req.computed + req.scheduled):
        logical_block, offset = divmod(pos, block_size)
        out.append(req.blocks[logical_block] * block_size + offset)
    return np.array(out, dtype=np.int64)


def write(cache: np.ndarray, new_rows: np.ndarray, slot_mapping: np.ndarray) -> np.ndarray:
    """Return a copy of ``cache`` with ``new_rows[t]`` stored at slot
    ``slot_mapping[t]``; negative slots (padding tokens) are skipped and every
    other slot keeps its old contents.

    ``cache`` is [num_blocks, block_size, ...]; a slot addresses one row of the
    cache viewed as [num_blocks * block_size, ...].
    """
    out = cache.copy()
    flat = out.reshape((-1,) + cache.shape[2:])
    for t, slot in enumerate(slot_mapping):
        if slot >= 0:
            flat[int(slot)] = new_rows[t]
    return out

"""Runner-side flat-batch metadata for one step (host, numpy).

"Model execution", section "Flattening a step": the runner concatenates the
scheduled tokens of all requests into one flat batch and hands the attention
layer ``query_start_loc`` (cumulative token offsets), ``seq_lens`` (context
after this step), ``block_table`` (physical block IDs per request) and
``slot_mapping`` (physical slot block_id * block_size + offset of each new
token).  These arrays are the inputs of ``pkv_write`` and
``pkv_attention_varlen``; they are built on the host, copied to the device
asynchronously, and never read back ("The runner must not synchronize").
"""

from __future__ import annotations

import numpy as np


def build(requests, block_size: int = 16, max_blocks_per_seq: int | None = None) -> dict:
    """Flatten a schedule.

    ``requests``: objects with ``computed`` (tokens already cached),
    ``scheduled`` (new tokens this step) and ``blocks`` (block table).
    Returns int32 ``query_start_loc`` / ``seq_lens`` / ``block_table`` (rows
    padded with block 0), int64 ``slot_mapping`` and the host scalars
    ``num_tokens``, ``max_query_len`` and ``max_seq_len``.
    """
    computed = np.array([r.computed for r in requests], dtype=np.int64)
    scheduled = np.array([r.scheduled for r in requests], dtype=np.int64)
    qsl = np.zeros(len(requests) + 1, dtype=np.int64)
    np.cumsum(scheduled, out=qsl[1:])
    seq_lens = computed + scheduled
    width = max_blocks_per_seq or max([len(r.blocks) for r in requests] + [1])
    table = np.zeros((len(requests), width), dtype=np.int32)
    for i, r in enumerate(requests):
        table[i, :len(r.blocks)] = r.blocks
    # new token k of request i sits at position computed[i] + k
    req_of_token = np.repeat(np.arange(len(requests)), scheduled)
    pos = np.arange(int(qsl[-1]), dtype=np.int64) - qsl[:-1][req_of_token] + computed[req_of_token]
    slot = table[req_of_token, pos // block_size].astype(np.int64) * block_size + pos % block_size
    return {
        "query_start_loc": qsl.astype(np.int32),
        "seq_lens": seq_lens.astype(np.int32),
        "block_table": table,
        "slot_mapping": slot,
        "positions": pos,
        "num_tokens": int(qsl[-1]),
        "max_query_len": int(scheduled.max()) if len(requests) else 0,
        "max_seq_len": int(seq_lens.max()) if len(requests) else 0,
    }


def context_slot_mapping(requests, block_size: int = 16) -> np.ndarray:
    """Slots of every context position 0..seq_len-1 of every request, in order
    (used to place cached-prefix K/V with ``pkv_write``)."""
    out = []
    for r in requests:
        pos = np.arange(r.computed + r.scheduled, dtype=np.int64)
        blocks = np.asarray(r.blocks, dtype=np.int64)
        out.append(blocks[pos // block_size] * block_size + pos % block_size)
    return np.concatenate(out) if out else np.zeros(0, dtype=np.int64)


def build_native(requests, block_size: int = 16, max_blocks_per_seq: int | None = None) -> dict:
    """``build`` through the library's host builder (``pkv_build_metadata``,
    the same arrays for a C host)."""
    from . import _binding
    return _binding.pkv_build_metadata([r.computed for r in requests],
                                       [r.scheduled for r in requests],
                                       [list(r.blocks) for r in requests], block_size,
                                       max_blocks_per_seq)


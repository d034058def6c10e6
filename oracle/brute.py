"""Brute-force attention: materialise each request's whole masked score matrix.

This is the textbook computation that "Inside the engine: kernels, CUDA graphs
and the life of a request" (section "Never materialise the TxT matrix")
describes before tiling removes it: S = scale * Q K^T over the full [n, L]
matrix, -inf where the causal mask (or a sliding window) hides a key, a
row-wise softmax, then P V.
Used only on tiny inputs, as a second formulation for ``ref`` to agree with.
"""

from __future__ import annotations

import numpy as np
from scipy.special import softmax


def _as_f64(x, dtype):
    if dtype == "bf16":
        bits = np.asarray(x, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def attention(q, k_cache, v_cache, query_start_loc, seq_lens, block_table, *,
              num_q_heads, num_kv_heads, softmax_scale, causal=True, block_size=16,
              dtype="f32", window=0):
    Q = _as_f64(q, dtype)
    Kc = _as_f64(k_cache, dtype).reshape(-1, num_kv_heads, Q.shape[2])
    Vc = _as_f64(v_cache, dtype).reshape(-1, num_kv_heads, Q.shape[2])
    out = np.zeros_like(Q)
    for r, L in enumerate(seq_lens):
        a, b = int(query_start_loc[r]), int(query_start_loc[r + 1])
        n, L = b - a, int(L)
        if n == 0:
            continue
        # physical slot of each logical key, block by block
        slots = []
        for blk in range(-(-L // block_size)):
            base = int(block_table[r][blk]) * block_size
            slots.extend(range(base, base + block_size))
        slots = np.array(slots[:L], dtype=np.int64)
        for h in range(num_q_heads):
            kvh = h * num_kv_heads // num_q_heads
            S = softmax_scale * Q[a:b, h, :] @ Kc[slots, kvh, :].T          # [n, L]
            if causal:
                # query i (0-based among the n new tokens) is token L - n + i
                S = np.where(np.tril(np.ones((n, L), dtype=bool), k=L - n), S, -np.inf)
            if window > 0:
                # sliding window: query i drops keys more than window - 1 behind it
                S = np.where(np.triu(np.ones((n, L), dtype=bool), k=L - n - window + 1), S,
                             -np.inf)
            P = softmax(S, axis=1)
            out[a:b, h, :] = P @ Vc[slots, kvh, :]
    return out

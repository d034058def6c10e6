"""Exact paged attention in float64: the two-pass definition, row by row.

Follows "Inside the engine: kernels, CUDA graphs and the life of a request":

* section "Never materialise the TxT matrix" - attention is S = QK^T, a
  row-wise softmax, then a product with V;
* section "Attention over a block table, not a contiguous tensor" - keys and
  values of a request live in 16-token blocks named by its block table;

and "Model execution", section "Flattening a step" - the new tokens of request
r are rows ``query_start_loc[r] .. query_start_loc[r+1]-1`` of the flat batch
and ``seq_lens[r]`` is its context after this step.

Readings taken where the pages are silent:

* the new tokens are the last n of the request's L context tokens, so new row i
  sits at position p = L - n + i and, under the causal mask, sees keys 0..p;
* query head h reads kv head h // (Hq / Hkv) (contiguous GQA groups);
* the cache is two tensors [num_blocks, block_size, Hkv, D] (K and V), i.e.
  one row of Hkv * D values per slot;
* a sliding window W > 0 ("Anatomy of a serving engine", section "Where it
  breaks", names sliding-window attention as a backend-dependent variant and
  gives no definition) keeps, for the row at position p, only keys j with
  j > p - W: the W most recent positions, the row's own included.

For every (row, head) the oracle takes pass 1, m = max_j s_j and
l = sum_j exp(s_j - m), then pass 2, o = sum_j (exp(s_j - m) / l) v_j, and
lse = m + ln l (natural log).  Rows of a chunk are processed together with
numpy, each with its own visible-key count.
"""

from __future__ import annotations

import numpy as np


def upcast(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of each element (bf16 arrays hold raw 16-bit patterns)."""
    if dtype == "bf16":
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if dtype == "f32":
        return x.astype(np.float64)
    raise ValueError(dtype)


def gather(cache: np.ndarray, table_row, seq_len: int, block_size: int) -> np.ndarray:
    """Logical rows 0..seq_len-1 of one request: row j is physical slot
    ``table_row[j // block_size] * block_size + j % block_size``."""
    flat = cache.reshape((-1,) + cache.shape[2:])
    j = np.arange(seq_len)
    blocks = np.asarray(table_row, dtype=np.int64)[j // block_size]
    return flat[blocks * block_size + j % block_size]


def attention(q, k_cache, v_cache, query_start_loc, seq_lens, block_table, *,
              num_q_heads: int, num_kv_heads: int, softmax_scale: float,
              causal: bool = True, block_size: int = 16, dtype: str = "f32",
              tokens=None, row_chunk: int = 512, kv_dtype: str | None = None,
              k_scale: float = 1.0, v_scale: float = 1.0, window: int = 0):
    """Attention output of the flat batch.

    With ``kv_dtype="e4m3"`` the caches hold 8-bit E4M3 codes and a cached K
    (V) element is ``k_scale`` (``v_scale``) times the code's value
    (``oracle.fp8``); q stays in ``dtype``.  ``window`` > 0 hides every key
    j <= p - window from the row at position p (on top of the causal mask).

    Returns ``(o, lse)``: o float64 [N, Hq, D], lse float64 [N, Hq].  With
    ``tokens`` (an iterable of flat-batch indices) only those rows are
    computed and every other entry is NaN.  A row that sees no key (empty
    causal range) gets o = 0 and lse = -inf.
    """
    qf = upcast(np.asarray(q), dtype)
    n_tok, hq, d = qf.shape
    assert hq == num_q_heads and hq % num_kv_heads == 0
    group = hq // num_kv_heads
    o = np.full((n_tok, hq, d), np.nan)
    lse = np.full((n_tok, hq), np.nan)
    wanted = None if tokens is None else np.zeros(n_tok, dtype=bool)
    if wanted is not None:
        wanted[np.asarray(list(tokens), dtype=np.int64)] = True
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    for r in range(len(seq_lens)):
        start, end = int(qsl[r]), int(qsl[r + 1])
        n, L = end - start, int(seq_lens[r])
        rows = np.arange(n)
        if wanted is not None:
            rows = rows[wanted[start:end]]
        if rows.size == 0:
            continue
        if kv_dtype == "e4m3":
            from . import fp8
            K = k_scale * fp8.decode(gather(k_cache, block_table[r], L, block_size))
            V = v_scale * fp8.decode(gather(v_cache, block_table[r], L, block_size))
        else:
            K = upcast(gather(k_cache, block_table[r], L, block_size), dtype)   # [L, Hkv, D]
            V = upcast(gather(v_cache, block_table[r], L, block_size), dtype)
        for c0 in range(0, rows.size, row_chunk):
            ri = rows[c0:c0 + row_chunk]
            pos = L - n + ri                                  # position of each row
            visible = pos + 1 if causal else np.full(ri.shape, L)
            mask = np.arange(L)[None, :] < visible[:, None]   # [rows, L]
            if window > 0:
                mask &= np.arange(L)[None, :] > (pos - window)[:, None]
            for h in range(hq):
                g = h // group
                s = softmax_scale * (qf[start + ri, h, :] @ K[:, g, :].T)   # [rows, L]
                s = np.where(mask, s, -np.inf)
                m = s.max(axis=1) if L > 0 else np.full(ri.shape, -np.inf)  # pass 1
                has = np.isfinite(m)
                m_safe = np.where(has, m, 0.0)
                e = np.where(mask, np.exp(s - m_safe[:, None]), 0.0)
                l = e.sum(axis=1)
                with np.errstate(invalid="ignore", divide="ignore"):
                    w = np.where(has[:, None], e / np.where(has, l, 1.0)[:, None], 0.0)
                o[start + ri, h, :] = w @ V[:, g, :] if L > 0 else 0.0          # pass 2
                with np.errstate(divide="ignore"):
                    lse[start + ri, h] = np.where(has, m_safe + np.log(np.where(has, l, 1.0)),
                                                  -np.inf)
    return o, lse


def paged_step(workload, tokens=None):
    """Oracle for one whole step of a workload: write the new K/V through the
    slot mapping, then attend.  Returns (o, lse, k_cache, v_cache, meta)."""
    from . import flatten as fl
    meta = fl.flatten(workload.requests, workload.block_size)
    kv = getattr(workload, "kv_dtype", None)
    k_new, v_new = workload.k_new, workload.v_new
    if kv == "e4m3":
        # the write stores each new element as the code of value / scale
        from . import fp8
        k_new = fp8.quantize(upcast(k_new, workload.dtype).astype(np.float32), workload.k_scale)
        v_new = fp8.quantize(upcast(v_new, workload.dtype).astype(np.float32), workload.v_scale)
    kc = fl.write(workload.k_pool, k_new, meta["slot_mapping"])
    vc = fl.write(workload.v_pool, v_new, meta["slot_mapping"])
    o, lse = attention(workload.q, kc, vc, meta["query_start_loc"], meta["seq_lens"],
                       meta["block_table"], num_q_heads=workload.num_q_heads,
                       num_kv_heads=workload.num_kv_heads,
                       softmax_scale=workload.softmax_scale, causal=workload.causal,
                       block_size=workload.block_size, dtype=workload.dtype, tokens=tokens,
                       kv_dtype=kv, k_scale=getattr(workload, "k_scale", 1.0),
                       v_scale=getattr(workload, "v_scale", 1.0),
                       window=getattr(workload, "window", 0))
    return o, lse, kc, vc, meta

"""Seeded synthetic inputs for paged KV attention.

This module only draws random numbers and lays them out as plain arrays.  It
holds none of the method's arithmetic: no slot or position arithmetic, no
softmax, no gather.  Both the float64 oracle (``oracle/``) and the CUDA path
(``paged_kv_attention_17_gb300``) consume what it returns, each turning the
schedule into kernel metadata with its own code.

A workload is the state a model runner hands to the attention layer for one
step ("Model execution", section "Flattening a step"):

* a schedule: per request, how many tokens are already in the cache
  (``computed``), how many are scheduled this step (``scheduled``) and its
  block table (physical block IDs of its context, in logical order);
* a KV pool of ``num_blocks`` blocks of 16 slots whose cached-prefix contents
  are random (prefix K/V are placed straight into the pool);
* Q, and the new tokens' K and V, for the flat batch of all scheduled tokens.

Values are N(0, 1) drawn from ``numpy.random.Generator(PCG64(seed))``; bf16
inputs are the float32 draws rounded to nearest-even bf16 and are stored as
their raw 16-bit patterns (numpy has no bf16 type).  Physical blocks are handed
out from ``rng.permutation(pool)``, context lengths from ``rng.integers``.

Named workloads follow the five shapes the attention pages are about: a tiny
three-request step like the pages' worked example, batch-1 long-context decode
(the FlashDecoding case), batched decode, a mixed chunked-prefill step and a
T = 8192 causal prefill.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16


@dataclass
class Request:
    """One request of a step: cached tokens, new tokens and block table."""

    computed: int
    scheduled: int
    blocks: list[int]


@dataclass
class Workload:
    name: str
    dtype: str                      # "f32" or "bf16"
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    num_blocks: int                 # pool size in blocks
    requests: list[Request]
    q: np.ndarray                   # [N, Hq, D]  float32 or uint16 (bf16 bits)
    k_new: np.ndarray               # [N, Hkv, D]
    v_new: np.ndarray               # [N, Hkv, D]
    k_pool: np.ndarray              # [num_blocks, 16, Hkv, D] (uint8 E4M3 codes for kv_dtype e4m3)
    v_pool: np.ndarray              # [num_blocks, 16, Hkv, D]
    softmax_scale: float
    causal: bool = True
    block_size: int = BLOCK_SIZE
    # Extra schedules with the same shape on disjoint blocks of the same pool
    # (index 0 is ``requests``); used to keep repeated timed steps L2-cold.
    replicas: list[list[Request]] = field(default_factory=list)
    kv_dtype: str | None = None     # None: caches in `dtype`; "e4m3": 8-bit codes + scales
    window: int = 0                 # > 0: sliding window of that many positions
    shared_blocks: int = 0          # leading blocks every request's table shares
    k_scale: float = 1.0
    v_scale: float = 1.0

    @property
    def num_tokens(self) -> int:
        return int(sum(r.scheduled for r in self.requests))

    @property
    def num_seqs(self) -> int:
        return len(self.requests)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); return the 16-bit patterns."""
    # uint32 arithmetic is exact for every finite input (only NaN patterns,
    # which a normal draw never produces, could wrap)
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def _values(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return x if dtype == "f32" else f32_to_bf16_bits(x)


def _codes(rng: np.random.Generator, shape) -> np.ndarray:
    # random 8-bit E4M3 codes: random sign, exponent field 4..8, any mantissa
    # (magnitudes 1/8 .. 3.75); drawn as bit fields, no rounding involved
    sign = rng.integers(0, 2, size=shape, dtype=np.uint8)
    exp = rng.integers(4, 9, size=shape, dtype=np.uint8)
    man = rng.integers(0, 8, size=shape, dtype=np.uint8)
    return (sign << 7) | (exp << 3) | man


def _blocks_needed(tokens: int, block_size: int) -> int:
    # number of whole blocks that hold `tokens` tokens (pool sizing only)
    return -(-tokens // block_size)


def _assign(perm: np.ndarray, start: int, shape: list[tuple[int, int]],
            block_size: int) -> tuple[list[Request], int]:
    reqs = []
    for computed, scheduled in shape:
        nb = _blocks_needed(computed + scheduled, block_size)
        reqs.append(Request(computed, scheduled, [int(b) for b in perm[start:start + nb]]))
        start += nb
    return reqs, start


def build(name: str, dtype: str, hq: int, hkv: int, d: int,
          shape: list[tuple[int, int]], seed: int = 0, pool_blocks: int | None = None,
          replicas: int = 1, scale: float | None = None, causal: bool = True,
          lengths_drawn: bool = False, rng: np.random.Generator | None = None,
          kv_dtype: str | None = None, k_scale: float = 1.0, v_scale: float = 1.0,
          window: int = 0) -> Workload:
    """Lay out a workload from a list of (computed, scheduled) pairs.

    The pool holds ``replicas`` disjoint copies of the schedule's blocks (or
    ``pool_blocks`` blocks if larger); the block IDs come from one random
    permutation of the pool.
    """
    rng = rng if rng is not None else np.random.Generator(np.random.PCG64(seed))
    need = sum(_blocks_needed(c + s, BLOCK_SIZE) for c, s in shape)
    num_blocks = max(need * replicas, pool_blocks or 0)
    perm = rng.permutation(num_blocks)
    reps, start = [], 0
    for _ in range(replicas):
        reqs, start = _assign(perm, start, shape, BLOCK_SIZE)
        reps.append(reqs)
    n = sum(s for _, s in shape)
    pool_shape = (num_blocks, BLOCK_SIZE, hkv, d)
    if kv_dtype == "e4m3":
        k_pool, v_pool = _codes(rng, pool_shape), _codes(rng, pool_shape)
    else:
        k_pool, v_pool = _values(rng, pool_shape, dtype), _values(rng, pool_shape, dtype)
    q = _values(rng, (n, hq, d), dtype)
    k_new = _values(rng, (n, hkv, d), dtype)
    v_new = _values(rng, (n, hkv, d), dtype)
    return Workload(name=name, dtype=dtype, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                    num_blocks=num_blocks, requests=reps[0], q=q, k_new=k_new, v_new=v_new,
                    k_pool=k_pool, v_pool=v_pool,
                    softmax_scale=float(scale if scale is not None else 1.0 / np.sqrt(d)),
                    causal=causal, replicas=reps, kv_dtype=kv_dtype, k_scale=float(k_scale),
                    v_scale=float(v_scale), window=int(window))


def build_cascade(name: str, dtype: str, hq: int, hkv: int, d: int, shared_blocks: int,
                  shape: list[tuple[int, int]], seed: int = 0, spare_blocks: int = 3,
                  rng: np.random.Generator | None = None, replicas: int = 1,
                  kv_dtype: str | None = None, k_scale: float = 1.0,
                  v_scale: float = 1.0) -> Workload:
    """Requests that share a prefix of ``shared_blocks`` blocks: each (c, s)
    pair is a request with c cached keys of its own after the prefix and s new
    tokens; its table is the shared blocks followed by its own.  Replicas
    repeat the batch on disjoint blocks (a prefix of their own each).
    kv_dtype "e4m3": the pools hold E4M3 codes (as ``build``)."""
    rng = rng if rng is not None else np.random.Generator(np.random.PCG64(seed))
    own = [_blocks_needed(c + s, BLOCK_SIZE) for c, s in shape]
    per_rep = shared_blocks + sum(own)
    num_blocks = per_rep * replicas + spare_blocks
    perm = rng.permutation(num_blocks)
    P = shared_blocks * BLOCK_SIZE
    reps, start = [], 0
    for _ in range(replicas):
        shared = [int(b) for b in perm[start:start + shared_blocks]]
        start += shared_blocks
        reqs = []
        for (c, s), nb in zip(shape, own):
            reqs.append(Request(P + c, s, shared + [int(b) for b in perm[start:start + nb]]))
            start += nb
        reps.append(reqs)
    n = sum(s for _, s in shape)
    pool_shape = (num_blocks, BLOCK_SIZE, hkv, d)
    if kv_dtype == "e4m3":
        k_pool, v_pool = _codes(rng, pool_shape), _codes(rng, pool_shape)
    else:
        k_pool, v_pool = _values(rng, pool_shape, dtype), _values(rng, pool_shape, dtype)
    q = _values(rng, (n, hq, d), dtype)
    k_new = _values(rng, (n, hkv, d), dtype)
    v_new = _values(rng, (n, hkv, d), dtype)
    return Workload(name=name, dtype=dtype, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                    num_blocks=num_blocks, requests=reps[0], q=q, k_new=k_new, v_new=v_new,
                    k_pool=k_pool, v_pool=v_pool, softmax_scale=float(1.0 / np.sqrt(d)),
                    replicas=reps, shared_blocks=shared_blocks, kv_dtype=kv_dtype,
                    k_scale=float(k_scale), v_scale=float(v_scale))


def cascade_64x4k(seed: int = 0, replicas: int = 1) -> Workload:
    """bf16, GQA 32/8, D = 128: 64 decodes sharing a 4096-token prefix (256
    blocks), each with U[0, 511] cached keys of its own and one new token."""
    rng = np.random.Generator(np.random.PCG64(seed))
    own = rng.integers(0, 512, size=64)
    return build_cascade("cascade_64x4k", "bf16", 32, 8, 128, 256, [(int(c), 1) for c in own],
                         rng=rng, replicas=replicas)


# ---------------------------------------------------------------------------
# The five named workloads.
# ---------------------------------------------------------------------------

def tiny_mixed_f32(seed: int = 0) -> Workload:
    """fp32, 2 q heads / 1 kv head, D = 64, 32-block pool: a 32-token prefill,
    a decode at context 40 and a 3-token cache-hit tail on a 45-token prefix."""
    return build("tiny_mixed_f32", "f32", 2, 1, 64, [(0, 32), (39, 1), (45, 3)],
                 seed=seed, pool_blocks=32)


def decode_8k(seed: int = 0, replicas: int = 1) -> Workload:
    """bf16 batch-1 decode at context 8192, GQA 32/8, D = 128; the block table is
    512 blocks of a randomly permuted 4096-block pool (8 disjoint replicas fit)."""
    assert 1 <= replicas <= 8
    return build("decode_8k", "bf16", 32, 8, 128, [(8191, 1)], seed=seed,
                 pool_blocks=4096, replicas=replicas)


def batched_decode_64(seed: int = 0, replicas: int = 1) -> Workload:
    """bf16, 64 decodes with context ~ U[512, 4096], GQA 32/8, D = 128."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = rng.integers(512, 4096 + 1, size=64)
    return build("batched_decode_64", "bf16", 32, 8, 128, [(int(c) - 1, 1) for c in ctx],
                 replicas=replicas, rng=rng)


def mixed_chunked(seed: int = 0, replicas: int = 1) -> Workload:
    """bf16 flat batch: a 2048-token prefill chunk on an empty prefix, a 3-token
    tail on a 1000-token prefix, then 62 decodes with context ~ U[256, 2048]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = rng.integers(256, 2048 + 1, size=62)
    shape = [(0, 2048), (1000, 3)] + [(int(c) - 1, 1) for c in ctx]
    return build("mixed_chunked", "bf16", 32, 8, 128, shape, replicas=replicas, rng=rng)


def prefill_8k(seed: int = 0, replicas: int = 1) -> Workload:
    """bf16 causal prefill of T = 8192 tokens, GQA 32/8, D = 128, written into
    512 shuffled 16-token blocks."""
    return build("prefill_8k", "bf16", 32, 8, 128, [(0, 8192)], seed=seed, replicas=replicas)


def batched_decode_64_e4m3(seed: int = 0, replicas: int = 1) -> Workload:
    """batched_decode_64 over an 8-bit E4M3 cache (k_scale = v_scale = 0.5)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = rng.integers(512, 4096 + 1, size=64)
    return build("batched_decode_64_e4m3", "bf16", 32, 8, 128, [(int(c) - 1, 1) for c in ctx],
                 replicas=replicas, rng=rng, kv_dtype="e4m3", k_scale=0.5, v_scale=0.5)


def decode_8k_e4m3(seed: int = 0, replicas: int = 1) -> Workload:
    """decode_8k over an 8-bit E4M3 cache (codes of magnitude 1/8 .. 3.75,
    k_scale = v_scale = 0.5): half the cache bytes per key, so the shuffled
    pool has 8192 blocks (268 MB, as decode_8k's) and 16 disjoint replicas fit."""
    assert 1 <= replicas <= 16
    return build("decode_8k_e4m3", "bf16", 32, 8, 128, [(8191, 1)], seed=seed,
                 pool_blocks=8192, replicas=replicas, kv_dtype="e4m3", k_scale=0.5,
                 v_scale=0.5)


def prefill_8k_e4m3(seed: int = 0, replicas: int = 1) -> Workload:
    """prefill_8k over an 8-bit E4M3 cache (k_scale = v_scale = 0.5): the
    8192 new tokens are quantised into the cache by the write, then attended."""
    return build("prefill_8k_e4m3", "bf16", 32, 8, 128, [(0, 8192)], seed=seed,
                 replicas=replicas, kv_dtype="e4m3", k_scale=0.5, v_scale=0.5)


NAMED = {
    "tiny_mixed_f32": tiny_mixed_f32,
    "decode_8k": decode_8k,
    "batched_decode_64": batched_decode_64,
    "mixed_chunked": mixed_chunked,
    "prefill_8k": prefill_8k,
    "decode_8k_e4m3": decode_8k_e4m3,
    "batched_decode_64_e4m3": batched_decode_64_e4m3,
    "prefill_8k_e4m3": prefill_8k_e4m3,
    "cascade_64x4k": cascade_64x4k,
}


def random_small(seed: int, dtype: str = "bf16", hq: int = 4, hkv: int = 2, d: int = 128,
                 num_seqs: int = 5, max_ctx: int = 200, max_new: int = 40,
                 causal: bool = True, spare_blocks: int = 7, kv_dtype: str | None = None,
                 k_scale: float = 1.0, v_scale: float = 1.0, window: int = 0) -> Workload:
    """A random small flat batch with ragged lengths (decodes, tails, prefills,
    empty requests) for parity sweeps."""
    rng = np.random.Generator(np.random.PCG64(seed))
    shape = []
    for _ in range(num_seqs):
        kind = int(rng.integers(0, 4))
        if kind == 0:                                  # decode
            c = int(rng.integers(0, max_ctx))
            shape.append((c, 1))
        elif kind == 1:                                # short tail on a prefix
            shape.append((int(rng.integers(0, max_ctx)), int(rng.integers(2, 5))))
        elif kind == 2:                                # prefill chunk
            shape.append((int(rng.integers(0, max_ctx // 2)), int(rng.integers(5, max_new + 1))))
        else:                                          # idle request (padding row)
            shape.append((int(rng.integers(0, max_ctx)), 0))
    need = sum(_blocks_needed(c + s, BLOCK_SIZE) for c, s in shape)
    return build(f"random_small_{seed}", dtype, hq, hkv, d, shape, rng=rng,
                 pool_blocks=need + spare_blocks, causal=causal, kv_dtype=kv_dtype,
                 k_scale=k_scale, v_scale=v_scale, window=window)

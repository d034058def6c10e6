"""Pins for the float64 oracle (CPU only).

Each test ties the oracle to something other than itself: the values the
pages print, torch's float64 scaled-dot-product attention on the contiguous
equivalent (a library routine with GQA and lower-right causal masking), closed
forms, and the invariances the pages state.  The last tests plant mistakes in
the oracle and check that a pin catches each one.
"""

import json
import math
import os
from types import SimpleNamespace

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from torch.nn.attention.bias import causal_lower_right

import workloads
from oracle import brute, flatten, merge, ref


def _req(c, s, blocks):
    return SimpleNamespace(computed=c, scheduled=s, blocks=list(blocks))


# --------------------------------------------------------------------------
# Flat-batch metadata: the printed example and the exercise
# --------------------------------------------------------------------------

def test_flatten_matches_printed_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "flatten_example.json")))
    reqs = [_req(r["computed"], r["scheduled"], r["blocks"]) for r in g["schedule"]]
    meta = flatten.flatten(reqs, g["block_size"])
    for key, want in g["printed"].items():
        assert meta[key].tolist() == want, key


def test_flatten_exercise_crosses_block(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "flatten_exercise.json")))
    r = g["request"]
    meta = flatten.flatten([_req(r["computed"], r["scheduled"], r["blocks"])], g["block_size"])
    assert meta["positions"].tolist() == g["expected"]["positions"]
    assert meta["slot_mapping"].tolist() == g["expected"]["slot_mapping"]
    assert meta["seq_lens"].tolist() == [g["expected"]["seq_len"]]


def test_write_places_rows_and_skips_padding():
    rng = np.random.default_rng(3)
    cache = rng.standard_normal((6, 16, 2, 4))
    new = rng.standard_normal((5, 2, 4))
    slots = np.array([17, -1, 0, 95, 40])
    out = flatten.write(cache, new, slots)
    flat_in, flat_out = cache.reshape(96, 2, 4), out.reshape(96, 2, 4)
    # written rows: block 1 offset 1, block 0 offset 0, block 5 offset 15, block 2 offset 8
    assert np.array_equal(out[1, 1], new[0]) and np.array_equal(out[0, 0], new[2])
    assert np.array_equal(out[5, 15], new[3]) and np.array_equal(out[2, 8], new[4])
    untouched = np.ones(96, bool)
    untouched[[17, 0, 95, 40]] = False
    assert np.array_equal(flat_in[untouched], flat_out[untouched])
    assert np.array_equal(cache.reshape(96, 2, 4), flat_in)   # input not modified


def test_write_then_gather_roundtrip():
    # every context position written through its slot comes back, in order,
    # through the block table
    req = _req(0, 37, [4, 0, 2])
    cache = np.zeros((5, 16, 1, 3))
    rows = np.arange(37 * 3, dtype=np.float64).reshape(37, 1, 3)
    meta = flatten.flatten([req])
    out = flatten.write(cache, rows, meta["slot_mapping"])
    back = ref.gather(out, meta["block_table"][0], 37, 16)
    assert np.array_equal(back, rows)
    assert np.array_equal(out[1], np.zeros((16, 1, 3)))  # unused block untouched


def test_bf16_upcast_exact():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000, 0x7F7F], dtype=np.uint16)
    got = ref.upcast(bits, "bf16")
    want = [1.0, -2.0, 1.0078125, 0.0, -0.0, 3.3895313892515355e38]
    assert got.tolist() == want
    # and the generator's rounding is nearest-even
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9], dtype=np.float32)
    assert workloads.f32_to_bf16_bits(x).tolist() == [0x3F80, 0x3F82, 0x3F80]


# --------------------------------------------------------------------------
# Attention against a library routine on the contiguous equivalent
# --------------------------------------------------------------------------

def _contiguous_case(rng, hq, hkv, d, shape):
    """Requests on an identity block table: the pool, read in order, is the
    contiguous K/V of each request."""
    reqs, blk = [], 0
    for c, s in shape:
        nb = -(-(c + s) // 16)
        reqs.append(_req(c, s, range(blk, blk + nb)))
        blk += nb
    nblk = max(blk, 1)
    kc = rng.standard_normal((nblk, 16, hkv, d))
    vc = rng.standard_normal((nblk, 16, hkv, d))
    n = sum(s for _, s in shape)
    q = rng.standard_normal((n, hq, d))
    return reqs, kc, vc, q


def _sdpa(q, kc, vc, reqs, hq, hkv, scale, causal):
    """torch float64 SDPA per request on contiguous K/V."""
    out = np.zeros_like(q)
    kflat = torch.from_numpy(kc.reshape(-1, hkv, kc.shape[-1]))
    vflat = torch.from_numpy(vc.reshape(-1, hkv, vc.shape[-1]))
    t0 = 0
    for r in reqs:
        n, L = r.scheduled, r.computed + r.scheduled
        if n == 0:
            continue
        base = r.blocks[0] * 16
        Q = torch.from_numpy(q[t0:t0 + n]).permute(1, 0, 2)[None]
        K = kflat[base:base + L].permute(1, 0, 2)[None]
        V = vflat[base:base + L].permute(1, 0, 2)[None]
        mask = causal_lower_right(n, L) if causal else None
        o = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale,
                                           enable_gqa=True)
        out[t0:t0 + n] = o[0].permute(1, 0, 2).numpy()
        t0 += n
    return out


def _ref(q, kc, vc, reqs, hq, hkv, scale, causal, **kw):
    meta = flatten.flatten(reqs)
    return ref.attention(q, kc, vc, meta["query_start_loc"], meta["seq_lens"],
                         meta["block_table"], num_q_heads=hq, num_kv_heads=hkv,
                         softmax_scale=scale, causal=causal, dtype="f32", **kw)


@pytest.mark.parametrize("hq,hkv,d", [(2, 1, 64), (4, 2, 16), (8, 2, 32), (3, 3, 8)])
@pytest.mark.parametrize("causal", [True, False])
def test_ref_matches_torch_sdpa(hq, hkv, d, causal):
    rng = np.random.default_rng(hq * 100 + d)
    shape = [(0, 32), (39, 1), (45, 3), (5, 11), (17, 16), (0, 1)]
    reqs, kc, vc, q = _contiguous_case(rng, hq, hkv, d, shape)
    scale = 1.0 / math.sqrt(d)
    o, lse = _ref(q, kc, vc, reqs, hq, hkv, scale, causal)
    want = _sdpa(q, kc, vc, reqs, hq, hkv, scale, causal)
    assert np.abs(o - want).max() < 1e-12


def test_ref_matches_brute_force_paged():
    w = workloads.random_small(11, dtype="f32", hq=4, hkv=2, d=16, num_seqs=6, max_ctx=70)
    meta = flatten.flatten(w.requests)
    o, _ = ref.attention(w.q, w.k_pool, w.v_pool, meta["query_start_loc"], meta["seq_lens"],
                         meta["block_table"], num_q_heads=4, num_kv_heads=2,
                         softmax_scale=w.softmax_scale, dtype="f32")
    b = brute.attention(w.q, w.k_pool, w.v_pool, meta["query_start_loc"], meta["seq_lens"],
                        meta["block_table"], num_q_heads=4, num_kv_heads=2,
                        softmax_scale=w.softmax_scale, dtype="f32")
    assert np.abs(o - b).max() < 1e-12


def test_bf16_path_matches_brute_force():
    w = workloads.random_small(5, dtype="bf16", hq=4, hkv=1, d=8, num_seqs=4, max_ctx=40)
    meta = flatten.flatten(w.requests)
    args = (w.q, w.k_pool, w.v_pool, meta["query_start_loc"], meta["seq_lens"],
            meta["block_table"])
    kw = dict(num_q_heads=4, num_kv_heads=1, softmax_scale=w.softmax_scale, dtype="bf16")
    o, _ = ref.attention(*args, **kw)
    assert np.abs(o - brute.attention(*args, **kw)).max() < 1e-12


# --------------------------------------------------------------------------
# Closed forms and stated invariants
# --------------------------------------------------------------------------

# --------------------------------------------------------------------------
# Sliding window (reading: row at position p keeps keys j > p - W)
# --------------------------------------------------------------------------

def _sdpa_window(q, kc, vc, reqs, hq, hkv, scale, window):
    """torch float64 SDPA with an explicit boolean band mask per request."""
    out = np.zeros_like(q)
    kflat = torch.from_numpy(kc.reshape(-1, hkv, kc.shape[-1]))
    vflat = torch.from_numpy(vc.reshape(-1, hkv, vc.shape[-1]))
    t0 = 0
    for r in reqs:
        n, L = r.scheduled, r.computed + r.scheduled
        if n == 0:
            continue
        base = r.blocks[0] * 16
        pos = torch.arange(L - n, L)[:, None]
        key = torch.arange(L)[None, :]
        mask = (key <= pos) & (key > pos - window)
        Q = torch.from_numpy(q[t0:t0 + n]).permute(1, 0, 2)[None]
        K = kflat[base:base + L].permute(1, 0, 2)[None]
        V = vflat[base:base + L].permute(1, 0, 2)[None]
        o = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale,
                                           enable_gqa=True)
        out[t0:t0 + n] = o[0].permute(1, 0, 2).numpy()
        t0 += n
    return out


@pytest.mark.parametrize("window", [1, 2, 7, 16, 17, 40, 1000])
def test_window_matches_torch_sdpa_band_mask(window):
    rng = np.random.default_rng(50 + window)
    shape = [(0, 32), (39, 1), (45, 3), (5, 11), (17, 16), (0, 1), (70, 2)]
    reqs, kc, vc, q = _contiguous_case(rng, 4, 2, 16, shape)
    o, _ = _ref(q, kc, vc, reqs, 4, 2, 0.25, True, window=window)
    want = _sdpa_window(q, kc, vc, reqs, 4, 2, 0.25, window)
    assert np.abs(o - want).max() < 1e-12


@pytest.mark.parametrize("window", [1, 5, 16, 33])
def test_window_matches_brute_force_paged(window):
    w = workloads.random_small(12, dtype="f32", hq=4, hkv=2, d=16, num_seqs=6, max_ctx=70)
    meta = flatten.flatten(w.requests)
    args = (w.q, w.k_pool, w.v_pool, meta["query_start_loc"], meta["seq_lens"],
            meta["block_table"])
    kw = dict(num_q_heads=4, num_kv_heads=2, softmax_scale=w.softmax_scale, dtype="f32",
              window=window)
    o, _ = ref.attention(*args, **kw)
    assert np.abs(o - brute.attention(*args, **kw)).max() < 1e-12


def test_window_of_one_returns_the_rows_own_value():
    rng = np.random.default_rng(7)
    reqs, kc, vc, q = _contiguous_case(rng, 4, 2, 16, [(20, 3), (0, 5)])
    o, lse = _ref(q, kc, vc, reqs, 4, 2, 0.25, True, window=1)
    vflat, kflat = vc.reshape(-1, 2, 16), kc.reshape(-1, 2, 16)
    t = 0
    for r in reqs:
        L, n = r.computed + r.scheduled, r.scheduled
        for i in range(n):
            slot = r.blocks[0] * 16 + L - n + i
            for h in range(4):
                assert np.array_equal(o[t, h], vflat[slot, h // 2])
                assert abs(lse[t, h] - 0.25 * q[t, h] @ kflat[slot, h // 2]) < 1e-12
            t += 1


def test_window_zero_query_gives_the_window_mean():
    rng = np.random.default_rng(8)
    reqs, kc, vc, q = _contiguous_case(rng, 2, 1, 8, [(40, 4), (3, 2)])
    q[:] = 0.0
    o, lse = _ref(q, kc, vc, reqs, 2, 1, 0.125, True, window=9)
    vflat = vc.reshape(-1, 1, 8)
    t = 0
    for r in reqs:
        L, n = r.computed + r.scheduled, r.scheduled
        for i in range(n):
            p = L - n + i
            lo = max(0, p - 9 + 1)
            base = r.blocks[0] * 16
            assert np.allclose(o[t, 0], vflat[base + lo:base + p + 1, 0].mean(axis=0),
                               atol=1e-13, rtol=0)
            assert abs(lse[t, 0] - math.log(p + 1 - lo)) < 1e-13
            t += 1


def test_window_equals_plain_attention_over_the_last_keys():
    # a decode row with window W sees exactly what a request holding only the
    # last W keys sees without a window (positions shift, the values do not)
    rng = np.random.default_rng(9)
    L, W = 77, 21
    reqs, kc, vc, q = _contiguous_case(rng, 4, 2, 16, [(L - 1, 1)])
    o, lse = _ref(q, kc, vc, reqs, 4, 2, 0.25, True, window=W)
    kf, vf = kc.reshape(-1, 2, 16), vc.reshape(-1, 2, 16)
    nb = -(-W // 16)
    k2 = np.zeros((nb * 16, 2, 16))
    v2 = np.zeros((nb * 16, 2, 16))
    k2[:W], v2[:W] = kf[L - W:L], vf[L - W:L]
    short = [_req(W - 1, 1, range(nb))]
    o2, lse2 = _ref(q, k2.reshape(nb, 16, 2, 16), v2.reshape(nb, 16, 2, 16), short, 4, 2,
                    0.25, True)
    assert np.abs(o - o2).max() < 1e-13 and np.abs(lse - lse2).max() < 1e-13


def test_zero_query_gives_prefix_mean_and_log_count():
    # all scores equal -> uniform weights over the visible keys
    rng = np.random.default_rng(1)
    shape = [(0, 20), (30, 3), (9, 1)]
    reqs, kc, vc, q = _contiguous_case(rng, 2, 1, 8, shape)
    q[:] = 0.0
    o, lse = _ref(q, kc, vc, reqs, 2, 1, 0.125, True)
    vflat = vc.reshape(-1, 1, 8)
    t = 0
    for r in reqs:
        L, n = r.computed + r.scheduled, r.scheduled
        base = r.blocks[0] * 16
        for i in range(n):
            visible = L - n + i + 1
            want = vflat[base:base + visible, 0].mean(axis=0)
            for h in range(2):
                assert np.allclose(o[t, h], want, atol=1e-13, rtol=0)
                assert abs(lse[t, h] - math.log(visible)) < 1e-13
            t += 1


def test_single_key_returns_its_value_exactly():
    # a first token (seq_len 1) and row 0 of a prefill see exactly one key
    rng = np.random.default_rng(2)
    reqs, kc, vc, q = _contiguous_case(rng, 4, 2, 16, [(0, 1), (0, 7)])
    o, lse = _ref(q, kc, vc, reqs, 4, 2, 0.25, True)
    vflat = vc.reshape(-1, 2, 16)
    for t, slot in ((0, reqs[0].blocks[0] * 16), (1, reqs[1].blocks[0] * 16)):
        for h in range(4):
            assert np.array_equal(o[t, h], vflat[slot, h // 2])


def test_gqa_head_mapping_with_head_constant_values():
    # V of kv head g is the constant g: query head h must return h // (Hq/Hkv)
    rng = np.random.default_rng(4)
    hq, hkv = 8, 4
    reqs, kc, vc, q = _contiguous_case(rng, hq, hkv, 4, [(12, 5), (0, 3)])
    vc[:] = np.arange(hkv, dtype=np.float64)[None, None, :, None]
    o, _ = _ref(q, kc, vc, reqs, hq, hkv, 0.5, True)
    for h in range(hq):
        assert np.allclose(o[:, h, :], h // (hq // hkv), atol=1e-13)


def test_paging_is_invisible_block_permutation_bit_identical():
    # "paging changes only the access pattern": move every block to a random
    # physical place and rewrite the tables; the oracle output is bit-identical
    rng = np.random.default_rng(5)
    shape = [(40, 3), (0, 33), (70, 1)]
    reqs, kc, vc, q = _contiguous_case(rng, 4, 2, 8, shape)
    o1, l1 = _ref(q, kc, vc, reqs, 4, 2, 0.3, True)
    nblk = kc.shape[0]
    perm = rng.permutation(nblk)          # logical block b moves to perm[b]
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    reqs2 = [_req(r.computed, r.scheduled, [int(perm[b]) for b in r.blocks]) for r in reqs]
    o2, l2 = _ref(q, kc2, vc2, reqs2, 4, 2, 0.3, True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_lse_matches_scipy_logsumexp():
    from scipy.special import logsumexp
    rng = np.random.default_rng(6)
    reqs, kc, vc, q = _contiguous_case(rng, 2, 2, 8, [(10, 4)])
    o, lse = _ref(q, kc, vc, reqs, 2, 2, 0.7, True)
    kflat = kc.reshape(-1, 2, 8)
    for i in range(4):
        for h in range(2):
            s = 0.7 * kflat[:10 + i + 1, h] @ q[i, h]
            assert abs(lse[i, h] - logsumexp(s)) < 1e-12


def test_token_subset_matches_full():
    w = workloads.random_small(8, dtype="bf16", hq=4, hkv=2, d=16, num_seqs=5)
    o_full, lse_full, *_ = ref.paged_step(w)
    sub = [0, w.num_tokens - 1, w.num_tokens // 2]
    o_sub, lse_sub, *_ = ref.paged_step(w, tokens=sub)
    # same rows, computed in a smaller batch: equal up to BLAS rounding order
    assert np.abs(o_sub[sub] - o_full[sub]).max() < 1e-14
    assert np.abs(lse_sub[sub] - lse_full[sub]).max() < 1e-14
    others = np.setdiff1d(np.arange(w.num_tokens), sub)
    assert np.isnan(o_sub[others]).all()


# --------------------------------------------------------------------------
# Online softmax, split-KV and merge against the two-pass reference
# --------------------------------------------------------------------------

@pytest.mark.parametrize("tile", [1, 3, 16, 64, 1000])
def test_online_softmax_equals_two_pass_and_m_only_rises(tile):
    rng = np.random.default_rng(tile)
    L, d = 300, 16
    s = rng.standard_normal(L) * 4.0
    v = rng.standard_normal((L, d))
    o, lse, trace = merge.online_softmax(s, v, tile)
    e = np.exp(s - s.max())
    assert np.abs(o - (e / e.sum()) @ v).max() < 1e-12
    assert abs(lse - (s.max() + math.log(e.sum()))) < 1e-12
    assert all(b >= a for a, b in zip(trace, trace[1:]))


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 19, 64])
def test_split_kv_merge_changes_nothing(splits):
    rng = np.random.default_rng(splits)
    L, d = 517, 8                             # ragged last block, some empty splits
    s = rng.standard_normal(L) * 3.0
    v = rng.standard_normal((L, d))
    o, lse = merge.split_attention_row(s, v, splits)
    e = np.exp(s - s.max())
    assert np.abs(o - (e / e.sum()) @ v).max() < 1e-12
    assert abs(lse - (s.max() + math.log(e.sum()))) < 1e-12


def test_split_ranges_cover_keys_once():
    for L in (0, 1, 15, 16, 17, 8192, 517):
        for S in (1, 2, 5, 64):
            rs = merge.split_ranges(L, S)
            covered = [j for a, b in rs for j in range(a, b)]
            assert covered == list(range(L))
            assert all(a % 16 == 0 for a, b in rs if b > a)


# --------------------------------------------------------------------------
# Planted mistakes: each must be caught by a pin above
# --------------------------------------------------------------------------

def _sdpa_pin_holds(hq=4, hkv=2, d=8, causal=True):
    rng = np.random.default_rng(77)
    reqs, kc, vc, q = _contiguous_case(rng, hq, hkv, d, [(5, 3), (0, 9), (20, 1)])
    o, _ = _ref(q, kc, vc, reqs, hq, hkv, 1 / math.sqrt(d), causal)
    want = _sdpa(q, kc, vc, reqs, hq, hkv, 1 / math.sqrt(d), causal)
    return np.abs(o - want).max() < 1e-12


def test_planted_gather_off_by_one_is_caught(monkeypatch):
    assert _sdpa_pin_holds()
    orig = ref.gather

    def shifted(cache, table_row, seq_len, block_size):
        rows = orig(cache, table_row, seq_len + 1, block_size)
        return rows[1:]
    monkeypatch.setattr(ref, "gather", shifted)
    assert not _sdpa_pin_holds()


def test_planted_k_v_swap_is_caught(monkeypatch):
    orig = ref.attention

    def swapped(q, k, v, *a, **kw):
        return orig(q, v, k, *a, **kw)
    monkeypatch.setattr(ref, "attention", swapped)
    assert not _sdpa_pin_holds()


def test_planted_upcast_error_is_caught(monkeypatch):
    orig = ref.upcast
    monkeypatch.setattr(ref, "upcast", lambda x, dt: orig(x, dt) * (1 + 1e-6))
    assert not _sdpa_pin_holds()


def _window_pin_holds(window=7):
    rng = np.random.default_rng(78)
    reqs, kc, vc, q = _contiguous_case(rng, 4, 2, 8, [(20, 3), (0, 9), (40, 1)])
    o, _ = _ref(q, kc, vc, reqs, 4, 2, 0.3, True, window=window)
    want = _sdpa_window(q, kc, vc, reqs, 4, 2, 0.3, window)
    return np.abs(o - want).max() < 1e-12


def test_planted_window_off_by_one_is_caught(monkeypatch):
    assert _window_pin_holds()
    orig = ref.attention

    def wider(*a, window=0, **kw):                # keeps j >= p - W: one key too many
        return orig(*a, window=window + 1 if window else 0, **kw)
    monkeypatch.setattr(ref, "attention", wider)
    assert not _window_pin_holds()


def test_planted_window_ignored_is_caught(monkeypatch):
    orig = ref.attention
    monkeypatch.setattr(ref, "attention", lambda *a, window=0, **kw: orig(*a, **kw))
    assert not _window_pin_holds()

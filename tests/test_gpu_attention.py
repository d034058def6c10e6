"""pkv_attention_varlen on the GPU against the float64 oracle.

Acceptance: max |err| <= 1e-2 and mean |err| <= 1e-3 for bf16 inputs with
fp32 accumulation (output rounded to bf16); fp32 inputs are held to 1e-4 /
1e-5.  Small workloads are compared element by element; the full-size
workloads run in the configuration the benchmark times (automatic split count)
and are compared on every row (decode_8k, batched_decode_64, mixed_chunked and
prefill_8k all fit the float64 oracle's budget).
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import ref
from tests.harness import device_inputs, errors, run_step

import paged_kv_attention_17_gb300 as pkv

pytestmark = pytest.mark.gpu

TOL = {"bf16": (1e-2, 1e-3), "f32": (1e-4, 1e-5)}


def _check(out, o_ref, dtype, tokens=None):
    mx, mean = errors(out, o_ref, tokens)
    tmax, tmean = TOL[dtype]
    assert mx <= tmax and mean <= tmean, (mx, mean)
    return mx, mean


def _check_lse(lse, lse_ref, tokens=None):
    got = lse.cpu().double().numpy()
    if tokens is not None:
        got, lse_ref = got[tokens], lse_ref[tokens]
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.abs(got[fin] - lse_ref[fin]).max() <= 1e-3


# --------------------------------------------------------------------------
# Small ragged batches: every element
# --------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("dtype,hq,hkv,d", [
    ("bf16", 8, 2, 128), ("bf16", 4, 4, 64), ("bf16", 32, 8, 128), ("f32", 2, 1, 64),
    ("f32", 4, 1, 128), ("bf16", 16, 1, 128)])
def test_random_small_batches(seed, dtype, hq, hkv, d):
    w = workloads.random_small(seed, dtype=dtype, hq=hq, hkv=hkv, d=d, num_seqs=6)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    _check(out, o_ref, dtype)
    _check_lse(lse, lse_ref)


@pytest.mark.parametrize("seed", range(4))
def test_non_causal(seed):
    w = workloads.random_small(seed + 40, dtype="bf16", hq=8, hkv=2, d=128, causal=False)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref, "bf16")
    _check_lse(lse, lse_ref)


def test_tiny_mixed_f32_every_element():
    w = workloads.tiny_mixed_f32()
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref, "f32")
    _check_lse(lse, lse_ref)


# --------------------------------------------------------------------------
# Full-size workloads in the benchmark's launch configuration
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["decode_8k", "batched_decode_64"])
def test_full_size_decode_all_rows(name):
    w = workloads.NAMED[name]()
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref, "bf16")
    _check_lse(lse, lse_ref)


def test_full_size_mixed_chunked_all_rows():
    # every row of the step: the 2048-token chunk, the 3-token tail, 62 decodes
    w = workloads.mixed_chunked()
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref, "bf16")
    _check_lse(lse, lse_ref)


def test_full_size_prefill_8k_all_rows():
    # all 8192 rows x 32 heads (about a minute of float64 oracle time)
    w = workloads.prefill_8k()
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref, "bf16")
    _check_lse(lse, lse_ref)


# --------------------------------------------------------------------------
# Invariances the pages state
# --------------------------------------------------------------------------

def test_split_count_changes_nothing():
    # "split-KV ... changes nothing about the result".  Outputs are bf16: two
    # split counts give fp32 results that differ by rounding only, and each is
    # then rounded to bf16 on its own, so two outputs may sit one bf16 step
    # apart (2^-7 of the largest magnitude) on top of the 1e-3 pairwise bound;
    # the fp32 LSEs are held to the plain 1e-3 pairwise bound, and the fp32
    # sweep below holds the outputs to it too.
    w = workloads.decode_8k()
    dev = device_inputs(w)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    outs, lses = [], []
    for s in (1, 2, 3, 7, 0, 64):
        out, lse, flag = run_step(dev, num_splits=s, write=(s == 1))
        assert int(flag.item()) == 0
        _check(out, o_ref, "bf16")
        _check_lse(lse, lse_ref)
        outs.append(out.float().cpu().numpy())
        lses.append(lse.cpu().numpy())
    for a in outs:
        for b in outs:
            assert np.abs(a - b).max() <= 1e-3 + 2 ** -7 * np.abs(a).max()
    for a in lses:
        for b in lses:
            assert np.abs(a - b).max() <= 1e-3


def test_split_count_changes_nothing_f32():
    # the same sweep with fp32 inputs and outputs: every pair of split counts
    # agrees to 1e-3 with no rounding allowance
    w = workloads.build("decode_8k_f32", "f32", 32, 8, 128, [(8191, 1)], seed=11,
                        pool_blocks=600)
    dev = device_inputs(w)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    outs = []
    for s in (1, 2, 3, 7, 0, 64):
        out, lse, flag = run_step(dev, num_splits=s, write=(s == 1))
        assert int(flag.item()) == 0
        _check(out, o_ref, "f32")
        _check_lse(lse, lse_ref)
        outs.append(out.cpu().numpy())
    for a in outs:
        for b in outs:
            assert np.abs(a - b).max() <= 1e-3


@pytest.mark.parametrize("num_seqs", [2, 37, 256, 257])
def test_longest_first_dispatch_unsplit(num_seqs):
    # An unsplit launch of 2..256 requests reads blockIdx.z as a rank of the
    # requests by decreasing seq_len; ties (equal lengths), idle requests (no
    # new token) and a prefill chunk in the batch must all keep their own
    # rows.  257 requests take the plain order.
    rng = np.random.Generator(np.random.PCG64(num_seqs))
    ctx = rng.choice([1, 16, 17, 200, 200, 513], size=num_seqs)
    shape = [(int(c) - 1, 1) for c in ctx]
    shape[0] = (0, 0)                        # idle request
    if num_seqs > 2:
        shape[1] = (40, 9)                   # a short prefill chunk
    w = workloads.build(f"lpt_{num_seqs}", "bf16", 8, 2, 128, shape, seed=num_seqs)
    dev = device_inputs(w)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    out, lse, flag = run_step(dev, num_splits=1)
    assert int(flag.item()) == 0
    _check(out, o_ref, "bf16")
    _check_lse(lse, lse_ref)


@pytest.mark.parametrize("hq,hkv", [(8, 4), (16, 2), (32, 4), (64, 8)])
@pytest.mark.parametrize("causal", [True, False])
def test_tensor_core_prefill_head_dim_64(hq, hkv, causal):
    # head_dim 64 with an even GQA group: long requests take the tensor-core
    # prefill (one 64-column half of each tile), beside decode rows and tails
    shape = [(0, 300), (500, 129), (40, 2), (1000, 1), (0, 1024), (77, 5)]
    w = workloads.build("d64_prefill", "bf16", hq, hkv, 64, shape, seed=hq + hkv, causal=causal)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref, "bf16")
    _check_lse(lse, lse_ref)


@pytest.mark.parametrize("window", [0, 200])
def test_tensor_core_prefill_head_dim_64_long_chunk(window):
    # a 2048-token chunk on a 1000-token prefix at GQA 32/8, every row
    w = workloads.build("d64_chunk", "bf16", 32, 8, 64, [(1000, 2048), (300, 1)], seed=64,
                        window=window)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref, "bf16")
    _check_lse(lse, lse_ref)


@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 128), (12, 4, 128), (15, 3, 64), (8, 8, 64)])
@pytest.mark.parametrize("causal", [True, False])
def test_tensor_core_prefill_odd_groups(hq, hkv, d, causal):
    # an odd GQA group (1, 3, 5): the tensor-core prefill pairs two query tiles
    # of one head; 1, 2, 3 and 9 tiles per request (the last pair half empty),
    # on empty and cached prefixes, beside decode rows
    shape = [(0, 100), (300, 256), (40, 300), (1000, 1), (0, 1100), (77, 5)]
    w = workloads.build("odd_group", "bf16", hq, hkv, d, shape, seed=hq * 3 + d, causal=causal)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref, "bf16")
    _check_lse(lse, lse_ref)


@pytest.mark.parametrize("window", [0, 300])
def test_tensor_core_prefill_odd_group_long_chunk(window):
    # MHA (group 1) at 32 heads: a 2048-token chunk on a 700-token prefix
    w = workloads.build("mha_chunk", "bf16", 32, 32, 128, [(700, 2048), (90, 1)], seed=7,
                        window=window)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref, "bf16")
    _check_lse(lse, lse_ref)


def test_split_heuristic_rule():
    # one wave of split CTAs over 7/8 of the decode CTA slots (two per SM for
    # the bf16 tensor-core build), at least 8 blocks per split, split off once
    # the grid is nearly full
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    target = 2 * sms * 7 // 8
    # batch 1, 8 KV heads, GQA group 4 (one 4-row tile): U = 8
    assert pkv.pkv_num_splits(1, 1, 8192, 32, 8, 128) == min(64, max(1, target // 8))
    # a short context caps the split at 8 blocks (128 keys) per split
    assert pkv.pkv_num_splits(1, 1, 300, 32, 8, 128) == 2
    # 64 decodes x 8 KV heads fill the device: no split
    assert pkv.pkv_num_splits(64, 1, 4096, 32, 8, 128) == 1


@pytest.mark.parametrize("seed", range(3))
def test_ragged_splits_first_block_speculation(seed):
    # each split's first blocks are loaded from the pre-launch table reading
    # for the split range max_seq_len would give, and kept only when the real
    # metadata confirms them: ragged lengths with several splits make the
    # ranges of all but the first split differ (the speculative fills wasted)
    w = workloads.random_small(60 + seed, dtype="bf16", hq=32, hkv=8, d=128, num_seqs=8,
                               max_ctx=1500)
    dev = device_inputs(w)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    for s in (2, 3, 5, 9):
        out, lse, flag = run_step(dev, num_splits=s, write=(s == 2))
        torch.cuda.synchronize()
        assert int(flag.item()) == 0
        _check(out, o_ref, "bf16")
        _check_lse(lse, lse_ref)


def test_block_permutation_is_bit_identical():
    # "paging changes only the access pattern": relocate every physical block
    # and rewrite the tables; with a fixed split count the result is identical
    w = workloads.random_small(21, dtype="bf16", hq=8, hkv=2, d=128, num_seqs=8, max_ctx=400)
    dev = device_inputs(w)
    out1, lse1, _ = run_step(dev, num_splits=3)
    perm = torch.from_numpy(np.random.default_rng(2).permutation(w.num_blocks)).cuda()
    kc2, vc2 = torch.empty_like(dev["k_cache"]), torch.empty_like(dev["v_cache"])
    kc2[perm] = dev["k_cache"]
    vc2[perm] = dev["v_cache"]
    dev2 = dict(dev, k_cache=kc2, v_cache=vc2, block_table=perm[dev["block_table"].long()].int())
    out2, lse2, _ = run_step(dev2, num_splits=3, write=False)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)


def test_single_key_returns_v_exactly():
    # a request whose first token is its whole context sees one key: out == v
    w = workloads.build("single", "bf16", 8, 2, 128, [(0, 1), (0, 1), (5, 1)], seed=3)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    v = dev["v_new"]
    for t in (0, 1):
        for h in range(8):
            assert torch.equal(out[t, h].view(torch.int16), v[t, h // 4].view(torch.int16))


def test_empty_and_idle_requests():
    w = workloads.build("idle", "bf16", 8, 2, 128, [(30, 0), (0, 0), (17, 2), (40, 0)], seed=4)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref, "bf16")
    # an empty batch enqueues nothing and succeeds
    e = torch.empty(0, 8, 128, dtype=torch.bfloat16, device="cuda")
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_attention_varlen(e, dev["k_cache"], dev["v_cache"], e, z, torch.zeros(0, dtype=torch.int32, device="cuda"),
                             dev["block_table"][:0], 0, 0, 0.1)


# --------------------------------------------------------------------------
# Data-dependent errors: flagged on the device, never a fault
# --------------------------------------------------------------------------

def test_bad_block_id_is_flagged():
    w = workloads.random_small(5, dtype="bf16", hq=8, hkv=2, d=128, num_seqs=4)
    dev = device_inputs(w)
    run_step(dev)
    bt = dev["block_table"].clone()
    bt[:, 0] = w.num_blocks + 1000
    dev2 = dict(dev, block_table=bt)
    out, lse, flag = run_step(dev2, write=False)
    torch.cuda.synchronize()
    assert int(flag.item()) & pkv.FLAG_BAD_BLOCK


def test_query_longer_than_context_is_flagged():
    w = workloads.build("bad", "bf16", 8, 2, 128, [(10, 3), (20, 1)], seed=6)
    dev = device_inputs(w)
    run_step(dev)
    sl = dev["seq_lens"].clone()
    sl[0] = 2                                        # q_len 3 > seq_len 2
    out, lse, flag = run_step(dict(dev, seq_lens=sl), write=False)
    torch.cuda.synchronize()
    assert int(flag.item()) & pkv.FLAG_BAD_LENGTHS


@pytest.mark.parametrize("new", [1, 8])
@pytest.mark.parametrize("splits", [0, 2])
def test_seq_len_beyond_table_row_is_flagged(new, splits):
    # a request whose seq_len needs more blocks than its table row holds is
    # flagged (decode kernel for one new token, prefill kernel for eight) and
    # skipped; max_seq_len stays within the row (the host rejects a larger
    # bound), so every table read, the pre-launch hints included, is in bounds
    w = workloads.build("narrow", "bf16", 8, 2, 128, [(40, 1), (20, new)], seed=8)
    dev = device_inputs(w)
    run_step(dev)
    torch.cuda.synchronize()
    width = int(dev["block_table"].shape[1])
    assert width == 3 and dev["meta"]["max_seq_len"] <= 16 * width
    sl = dev["seq_lens"].clone()
    sl[1] = 16 * width + 5                           # one block past the row
    out, lse, flag = run_step(dict(dev, seq_lens=sl), num_splits=splits, write=False)
    torch.cuda.synchronize()
    assert int(flag.item()) & pkv.FLAG_BAD_LENGTHS
    # the request that fits is still computed
    o_ref, lse_ref, *_ = ref.paged_step(w, tokens=[0])
    _check(out, o_ref, "bf16", [0])

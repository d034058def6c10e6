"""pkv_cascade_attention on the GPU against the float64 oracle.

Batches whose requests share a block-aligned prefix: the result must equal
plain paged attention over shared ++ own blocks (``ref.paged_step`` on the
full tables; ``oracle.cascade`` pins that this is also the two-level result),
within the attention tolerance (bf16 max 1e-2 / mean 1e-3, fp32 1e-4 / 1e-5).
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import ref
from tests.harness import device_inputs, errors

import paged_kv_attention_17_gb300 as pkv

pytestmark = pytest.mark.gpu

TOL = {"bf16": (1e-2, 1e-3), "f32": (1e-4, 1e-5)}


def cascade_inputs(w, device="cuda"):
    """Device tensors of a cascade workload: the plain inputs plus the shared
    table, the own-key tables and lengths."""
    d = device_inputs(w, device)
    P = w.shared_blocks * 16
    own = [r.blocks[w.shared_blocks:] for r in w.requests]
    width = max(max(len(b) for b in own), 1)
    table = np.zeros((len(own), width), dtype=np.int32)
    for i, b in enumerate(own):
        table[i, :len(b)] = b
    d["shared_table"] = torch.tensor(w.requests[0].blocks[:w.shared_blocks], dtype=torch.int32,
                                     device=device)
    d["suffix_table"] = torch.from_numpy(table).to(device)
    lens = [r.computed + r.scheduled - P for r in w.requests]
    d["suffix_lens"] = torch.tensor(lens, dtype=torch.int32, device=device)
    d["max_suffix_len"] = max(lens)
    return d


def run_cascade(d, prefix_splits=0, with_lse=True):
    w = d["w"]
    flag = torch.zeros(1, dtype=torch.int32, device=d["q"].device)
    pkv.pkv_write(d["k_new"], d["v_new"], d["slot_mapping"], d["k_cache"], d["v_cache"],
                  error_flag=flag)
    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device=d["q"].device) \
        if with_lse else None
    pkv.pkv_cascade_attention(d["q"], d["k_cache"], d["v_cache"], out, d["qsl"],
                              d["suffix_lens"], d["suffix_table"], d["shared_table"],
                              d["meta"]["max_query_len"], d["max_suffix_len"], w.softmax_scale,
                              prefix_splits=prefix_splits, lse_out=lse, error_flag=flag)
    return out, lse, flag


def _check(out, lse, w, dtype, tokens=None):
    o_ref, lse_ref, *_ = ref.paged_step(w, tokens=tokens)
    mx, mean = errors(out, o_ref, tokens)
    tmax, tmean = TOL[dtype]
    assert mx <= tmax and mean <= tmean, (mx, mean)
    got = lse.cpu().double().numpy()
    if tokens is not None:
        got, lse_ref = got[tokens], lse_ref[tokens]
    assert np.abs(got - lse_ref).max() <= 1e-3


@pytest.mark.parametrize("prefix_splits", [1, 3, 0])
@pytest.mark.parametrize("shared_blocks", [1, 5, 40])
@pytest.mark.parametrize("dtype,hq,hkv,d", [("bf16", 32, 8, 128), ("bf16", 8, 1, 64),
                                            ("f32", 4, 2, 128), ("bf16", 64, 8, 128),
                                            ("bf16", 16, 8, 128), ("bf16", 64, 4, 128),
                                            ("bf16", 12, 4, 128)])
def test_decode_batches(prefix_splits, shared_blocks, dtype, hq, hkv, d):
    # tensor-core prefix pass for bf16 / D 128 / groups 2, 4, 8, 16; CUDA-core
    # prefix pass for D 64, fp32 and group 3
    rng = np.random.Generator(np.random.PCG64(shared_blocks * 31 + hq))
    shape = [(int(c), 1) for c in rng.integers(0, 200, size=12)] + [(0, 1), (15, 1), (16, 1)]
    w = workloads.build_cascade("casc", dtype, hq, hkv, d, shared_blocks, shape, rng=rng)
    dev = cascade_inputs(w)
    out, lse, flag = run_cascade(dev, prefix_splits)
    assert int(flag.item()) == 0
    _check(out, lse, w, dtype)


@pytest.mark.parametrize("shape", [
    [(3, 2), (40, 4), (0, 3), (100, 1)],              # multi-token decode rows
    [(0, 9), (30, 20), (5, 1), (64, 70)],             # long own parts: CUDA-core tiles
])
def test_multi_token_requests(shape):
    w = workloads.build_cascade("casc_mt", "bf16", 16, 4, 128, 7, shape, seed=5)
    dev = cascade_inputs(w)
    out, lse, flag = run_cascade(dev)
    assert int(flag.item()) == 0
    _check(out, lse, w, "bf16")


def test_no_shared_prefix_is_plain_attention():
    w = workloads.build_cascade("casc0", "bf16", 8, 2, 128, 0, [(30, 1), (0, 2), (77, 1)],
                                seed=6)
    dev = cascade_inputs(w)
    out, lse, flag = run_cascade(dev)
    assert int(flag.item()) == 0
    _check(out, lse, w, "bf16")


def test_matches_the_plain_call_on_the_full_tables():
    rng = np.random.Generator(np.random.PCG64(77))
    shape = [(int(c), 1) for c in rng.integers(0, 300, size=20)]
    w = workloads.build_cascade("casc_eq", "bf16", 32, 8, 128, 64, shape, rng=rng)
    dev = cascade_inputs(w)
    out, _, _ = run_cascade(dev)
    plain = torch.empty_like(dev["q"])
    m = dev["meta"]
    pkv.pkv_attention_varlen(dev["q"], dev["k_cache"], dev["v_cache"], plain, dev["qsl"],
                             dev["seq_lens"], dev["block_table"], m["max_query_len"],
                             m["max_seq_len"], w.softmax_scale)
    # both round fp32 results of |o| < 1 to bf16: at most one ulp (2^-8) apart
    assert (out.float() - plain.float()).abs().max().item() <= 2.0 ** -8


def test_cascade_64x4k_sampled_rows():
    # the benchmark's batch: 64 decodes sharing a 4096-token prefix
    w = workloads.cascade_64x4k()
    dev = cascade_inputs(w)
    out, lse, flag = run_cascade(dev)
    assert int(flag.item()) == 0
    toks = [0, 1, 17, 31, 32, 62, 63]
    _check(out, lse, w, "bf16", toks)


def run_cascade_e4m3(d, prefix_splits=0):
    w = d["w"]
    flag = torch.zeros(1, dtype=torch.int32, device=d["q"].device)
    pkv.pkv_write_e4m3(d["k_new"], d["v_new"], d["slot_mapping"], d["k_cache"], d["v_cache"],
                       w.k_scale, w.v_scale, error_flag=flag)
    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device=d["q"].device)
    pkv.pkv_cascade_attention(d["q"], d["k_cache"], d["v_cache"], out, d["qsl"],
                              d["suffix_lens"], d["suffix_table"], d["shared_table"],
                              d["meta"]["max_query_len"], d["max_suffix_len"], w.softmax_scale,
                              prefix_splits=prefix_splits, lse_out=lse, error_flag=flag,
                              kv_scales=(w.k_scale, w.v_scale))
    return out, lse, flag


@pytest.mark.parametrize("prefix_splits", [1, 3, 0])
@pytest.mark.parametrize("shared_blocks", [1, 5, 40])
@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (8, 1, 64), (12, 4, 128)])
def test_cascade_over_e4m3_cache(prefix_splits, shared_blocks, hq, hkv, d):
    # pkv_cascade_attention_e4m3: the prefix pass on the CUDA-core tiles, the
    # own-key pass on the decode kernel, against plain attention over the
    # dequantised full tables
    rng = np.random.Generator(np.random.PCG64(shared_blocks * 17 + hq))
    shape = [(int(c), 1) for c in rng.integers(0, 200, size=12)] + [(0, 1), (15, 2), (16, 1)]
    w = workloads.build_cascade("casc_e4m3", "bf16", hq, hkv, d, shared_blocks, shape, rng=rng,
                                kv_dtype="e4m3", k_scale=0.6, v_scale=0.35)
    dev = cascade_inputs(w)
    out, lse, flag = run_cascade_e4m3(dev, prefix_splits)
    assert int(flag.item()) == 0
    _check(out, lse, w, "bf16")


def test_cascade_split_rule():
    # pkv_cascade_splits as the header states it: T = floor(7 SMs / 8); the
    # tensor-core pass (bf16, an even group dividing 128) over U = H_kv x
    # ceil(group x tokens / 256) row tiles with at least four 128-key tiles a
    # split, the CUDA-core pass over U = H_kv x ceil(group x tokens / 16) with
    # at least 8 blocks a split; max(1, min(T // U, length cap, 63))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T = sms * 7 // 8

    def rule(n, blocks, hq, hkv, tc):
        g = hq // hkv
        U = hkv * -(-(g * n) // (256 if tc else 16))
        cap = -(-blocks // 32) if tc else blocks // 8
        return max(1, min(T // U, cap, 63))

    cases = [  # (tokens, shared blocks, hq, hkv, dtype, tensor-core pass)
        (64, 256, 32, 8, torch.bfloat16, True),       # the bench batch: 8 splits
        (1, 4096, 32, 8, torch.bfloat16, True),       # a 64K-token prefix
        (2048, 1024, 32, 8, torch.bfloat16, True),    # a full grid: one split
        (64, 5, 32, 8, torch.bfloat16, True),         # under four tiles: one split
        (64, 256, 12, 4, torch.bfloat16, False),      # odd group: CUDA-core pass
        (64, 256, 32, 8, torch.float32, False),       # fp32: CUDA-core pass
        (64, 5, 32, 8, torch.float32, False),         # under 8 blocks: one split
        (3, 600, 8, 1, torch.bfloat16, True),         # group 8
    ]
    for n, blocks, hq, hkv, dt, tc in cases:
        assert pkv.pkv_cascade_splits(n, blocks, hq, hkv, 128, dt) == rule(n, blocks, hq, hkv, tc), \
            (n, blocks, hq, hkv, dt)
    assert pkv.pkv_cascade_splits(64, 0, 32, 8, 128) == 0


def test_cascade_e4m3_rejects_bad_scales():
    w = workloads.build_cascade("casc_e4m3_bad", "bf16", 8, 2, 128, 2, [(3, 1)], seed=1,
                                kv_dtype="e4m3", k_scale=0.5, v_scale=0.5)
    dev = cascade_inputs(w)
    out = torch.empty_like(dev["q"])
    with pytest.raises(pkv.PkvError):
        pkv.pkv_cascade_attention(dev["q"], dev["k_cache"], dev["v_cache"], out, dev["qsl"],
                                  dev["suffix_lens"], dev["suffix_table"], dev["shared_table"],
                                  dev["meta"]["max_query_len"], dev["max_suffix_len"],
                                  w.softmax_scale, kv_scales=(0.0, 0.5))

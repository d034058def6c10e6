"""pkv_write_attention_varlen on the GPU: the KV write folded into the decode
kernel for decode-class steps, and write + attention otherwise.

The cache after the call must equal the oracle's write bit for bit, the
output the float64 oracle within the attention tolerance, and the output
must be bit-identical to the two separate calls (the same arithmetic).
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import ref
from tests.harness import device_inputs, errors, run_fused_step, run_step

pytestmark = pytest.mark.gpu

TOL = {"bf16": (1e-2, 1e-3), "f32": (1e-4, 1e-5)}


def _cache_bits(t):
    if t.dtype == torch.uint8:
        return t.cpu().numpy()
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).cpu().numpy()


def _ref_bits(x, dtype):
    if x.dtype == np.uint8:
        return x
    return np.ascontiguousarray(x).view(np.int16 if dtype == "bf16" else np.int32)


def _check(w, dev, out, lse, flag, dtype, tokens=None):
    o_ref, lse_ref, kc, vc, _ = ref.paged_step(w, tokens=tokens)
    assert int(flag.item()) == 0
    mx, mean = errors(out, o_ref, tokens)
    assert mx <= TOL[dtype][0] and mean <= TOL[dtype][1], (mx, mean)
    got = lse.cpu().double().numpy()
    if tokens is not None:
        got, lse_ref = got[tokens], lse_ref[tokens]
    assert np.abs(got - lse_ref).max() <= 1e-3
    assert np.array_equal(_cache_bits(dev["k_cache"]), _ref_bits(kc, dtype))
    assert np.array_equal(_cache_bits(dev["v_cache"]), _ref_bits(vc, dtype))


@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("dtype,hq,hkv,d,qlen", [
    ("bf16", 32, 8, 128, 1), ("bf16", 32, 8, 128, 4), ("bf16", 8, 8, 64, 2),
    ("bf16", 64, 8, 128, 1), ("f32", 4, 1, 128, 3), ("bf16", 16, 1, 128, 1)])
def test_decode_batches(splits, dtype, hq, hkv, d, qlen):
    rng = np.random.Generator(np.random.PCG64(hq * 3 + qlen + d))
    ctx = rng.integers(0, 600, size=10)
    shape = [(int(c), qlen) for c in ctx] + [(0, qlen), (15, qlen), (16, qlen), (31, 1)]
    w = workloads.build("fused", dtype, hq, hkv, d, shape, rng=rng)
    dev = device_inputs(w)
    out, lse, flag = run_fused_step(dev, num_splits=splits)
    _check(w, dev, out, lse, flag, dtype)


def test_bit_identical_to_separate_calls():
    rng = np.random.Generator(np.random.PCG64(90))
    shape = [(int(c), int(n)) for c, n in zip(rng.integers(0, 900, size=16),
                                              rng.integers(1, 5, size=16))]
    w = workloads.build("fused_eq", "bf16", 32, 8, 128, shape, rng=rng)
    for splits in (1, 4, 0):
        dev = device_inputs(w)
        fused, lse_f, _ = run_fused_step(dev, num_splits=splits)
        kf, vf = dev["k_cache"].clone(), dev["v_cache"].clone()
        dev2 = device_inputs(w)
        sep, lse_s, _ = run_step(dev2, num_splits=splits)
        assert torch.equal(fused, sep) and torch.equal(lse_f, lse_s), splits
        assert torch.equal(kf, dev2["k_cache"]) and torch.equal(vf, dev2["v_cache"])


def test_mixed_step_takes_the_separate_write():
    w = workloads.random_small(300, hq=8, hkv=2, d=128, num_seqs=8, max_new=60)
    assert max(r.scheduled for r in w.requests) > 4
    dev = device_inputs(w)
    out, lse, flag = run_fused_step(dev)
    _check(w, dev, out, lse, flag, "bf16")


def test_decode_8k_full_size():
    w = workloads.decode_8k()
    dev = device_inputs(w)
    out, lse, flag = run_fused_step(dev)
    _check(w, dev, out, lse, flag, "bf16")


def test_padding_slot_is_not_stored_and_bad_slot_is_flagged():
    rng = np.random.Generator(np.random.PCG64(91))
    w = workloads.build("fused_pad", "bf16", 8, 2, 128, [(40, 2), (100, 1), (7, 3)], rng=rng)
    dev = device_inputs(w)
    pool_k = dev["k_cache"].clone()
    slots = dev["slot_mapping"].clone()
    slots[1] = -1                                  # second token of request 0: not stored
    dev["slot_mapping"] = slots
    out, lse, flag = run_fused_step(dev)
    assert int(flag.item()) == 0
    s_pad = int(dev["meta"]["slot_mapping"][1])
    kf = dev["k_cache"].view(-1, 2, 128)
    assert torch.equal(kf[s_pad], pool_k.view(-1, 2, 128)[s_pad])   # untouched
    s0 = int(dev["meta"]["slot_mapping"][0])
    assert torch.equal(kf[s0], dev["k_new"][0])                       # stored
    # a slot past the cache: skipped and flagged
    dev = device_inputs(w)
    slots = dev["slot_mapping"].clone()
    slots[3] = w.num_blocks * 16 + 5
    dev["slot_mapping"] = slots
    _, _, flag = run_fused_step(dev)
    assert int(flag.item()) & 2


@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("hq,hkv,d,qlen", [(32, 8, 128, 1), (32, 8, 128, 3), (16, 2, 64, 1),
                                           (64, 8, 128, 2)])
def test_e4m3_decode_batches(splits, hq, hkv, d, qlen):
    # the write quantises in the decode kernel: codes bit-exact to the oracle's
    rng = np.random.Generator(np.random.PCG64(hq * 5 + qlen + d))
    ctx = rng.integers(0, 600, size=10)
    shape = [(int(c), qlen) for c in ctx] + [(0, qlen), (15, qlen), (16, qlen)]
    w = workloads.build("fused8", "bf16", hq, hkv, d, shape, rng=rng, kv_dtype="e4m3",
                        k_scale=0.037, v_scale=1.9)
    dev = device_inputs(w)
    out, lse, flag = run_fused_step(dev, num_splits=splits)
    _check(w, dev, out, lse, flag, "bf16")


def test_e4m3_bit_identical_to_separate_calls():
    rng = np.random.Generator(np.random.PCG64(93))
    shape = [(int(c), int(n)) for c, n in zip(rng.integers(0, 900, size=12),
                                              rng.integers(1, 5, size=12))]
    w = workloads.build("fused8_eq", "bf16", 32, 8, 128, shape, rng=rng, kv_dtype="e4m3",
                        k_scale=0.5, v_scale=0.25)
    dev = device_inputs(w)
    fused, _, _ = run_fused_step(dev, num_splits=3)
    dev2 = device_inputs(w)
    sep, _, _ = run_step(dev2, num_splits=3)
    assert torch.equal(fused, sep)
    assert torch.equal(dev["k_cache"], dev2["k_cache"]) and torch.equal(dev["v_cache"],
                                                                        dev2["v_cache"])


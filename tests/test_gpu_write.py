"""pkv_write on the GPU: bit-exact against the oracle's scatter."""

import numpy as np
import pytest
import torch

import workloads
from oracle import flatten as oflat
from tests.harness import device_inputs

import paged_kv_attention_17_gb300 as pkv

pytestmark = pytest.mark.gpu


def _bits(t):
    return (t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)).cpu().numpy()


def _want_bits(x, dtype):
    return x.view(np.int16) if dtype == "bf16" else x.astype(np.float32).view(np.int32)


@pytest.mark.parametrize("name", ["tiny_mixed_f32", "decode_8k", "mixed_chunked", "prefill_8k"])
def test_write_bit_exact_named(name):
    w = workloads.NAMED[name]()
    d = device_inputs(w)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_write(d["k_new"], d["v_new"], d["slot_mapping"], d["k_cache"], d["v_cache"],
                  error_flag=flag)
    meta = oflat.flatten(w.requests)
    k_ref = oflat.write(w.k_pool, w.k_new, meta["slot_mapping"])
    v_ref = oflat.write(w.v_pool, w.v_new, meta["slot_mapping"])
    assert int(flag.item()) == 0
    assert np.array_equal(_bits(d["k_cache"]), _want_bits(k_ref, w.dtype))
    assert np.array_equal(_bits(d["v_cache"]), _want_bits(v_ref, w.dtype))


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("dtype,hkv,d", [("bf16", 2, 128), ("f32", 1, 64), ("bf16", 3, 64)])
def test_write_bit_exact_random_with_padding(seed, dtype, hkv, d):
    w = workloads.random_small(seed, dtype=dtype, hq=hkv * 2, hkv=hkv, d=d, num_seqs=7)
    dev = device_inputs(w)
    slots = dev["meta"]["slot_mapping"].copy()
    rng = np.random.default_rng(seed)
    pad = rng.random(slots.shape) < 0.3                 # padding tokens: slot -1
    slots[pad] = -1
    st = torch.from_numpy(slots).cuda()
    pkv.pkv_write(dev["k_new"], dev["v_new"], st, dev["k_cache"], dev["v_cache"])
    k_ref = oflat.write(w.k_pool, w.k_new, slots)
    v_ref = oflat.write(w.v_pool, w.v_new, slots)
    assert np.array_equal(_bits(dev["k_cache"]), _want_bits(k_ref, dtype))
    assert np.array_equal(_bits(dev["v_cache"]), _want_bits(v_ref, dtype))


def test_write_out_of_range_slot_is_flagged_and_skipped():
    w = workloads.random_small(3, num_seqs=4)
    dev = device_inputs(w)
    slots = dev["meta"]["slot_mapping"].copy()
    slots[0] = w.num_blocks * 16 + 5                    # beyond the cache
    before_k = _bits(dev["k_cache"]).copy()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_write(dev["k_new"], dev["v_new"], torch.from_numpy(slots).cuda(), dev["k_cache"],
                  dev["v_cache"], error_flag=flag)
    assert int(flag.item()) & pkv.FLAG_BAD_SLOT
    want = oflat.write(w.k_pool, w.k_new, np.where(np.arange(len(slots)) == 0, -1, slots))
    assert np.array_equal(_bits(dev["k_cache"]), _want_bits(want, w.dtype))
    assert before_k.shape == _bits(dev["k_cache"]).shape


def test_write_empty_batch_is_noop():
    k = torch.zeros(4, 16, 2, 128, dtype=torch.bfloat16, device="cuda")
    e = torch.zeros(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    pkv.pkv_write(e, e, torch.zeros(0, dtype=torch.int64, device="cuda"), k, k.clone())
    torch.cuda.synchronize()
    assert int(k.abs().sum().item()) == 0

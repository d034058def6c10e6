"""The allocation-free attention entry point.

pkv_attention_varlen_noalloc serves callers that cannot allocate device
memory (their memory belongs to another runtime's allocator, or they must not
block in cudaMalloc/cudaFree): the split-KV partials go to a fixed array
inside the library instead of a caller workspace.  These tests call it
through the C ABI and check, on two calls in a row (the array keeps the
previous call's contents), that it returns what the allocating entry point
returns, within the tolerance the parity tests use.  The file is collected
last so that a run stopping at the first failure has run every other test.
"""

import numpy as np
import pytest
import torch

import workloads
from tests.harness import device_inputs, run_step

pytestmark = pytest.mark.gpu


def _pkv():
    from paged_kv_attention_17_gb300 import build
    build.build()
    import paged_kv_attention_17_gb300 as pkv
    return pkv


@pytest.mark.parametrize("name", ["decode_8k", "mixed_chunked"])
def test_noalloc_matches_allocating_entry_point_twice(name):
    pkv = _pkv()
    w = workloads.NAMED[name]()
    dev = device_inputs(w)
    meta = dev["meta"]
    ref_out, ref_lse, flag = run_step(dev)                # workspace path
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    want = ref_out.float().cpu().numpy()
    splits = pkv.pkv_num_splits(w.num_seqs, meta["max_query_len"], meta["max_seq_len"],
                                w.num_q_heads, w.num_kv_heads, w.head_dim)
    if name == "decode_8k":
        assert splits > 1                                  # the scratch array is really used
    for _ in range(2):
        out = torch.full_like(dev["q"], float("nan"))
        lse = torch.full(dev["q"].shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        pkv.pkv_attention_varlen_noalloc(dev["q"], dev["k_cache"], dev["v_cache"], out, dev["qsl"],
                                         dev["seq_lens"], dev["block_table"], meta["max_query_len"],
                                         meta["max_seq_len"], w.softmax_scale, causal=w.causal,
                                         lse_out=lse, error_flag=flag)
        torch.cuda.synchronize()
        assert int(flag.item()) == 0
        got = out.float().cpu().numpy()
        err = np.abs(got - want)
        assert err.max() <= 1e-2 and err.mean() <= 1e-3, (err.max(), err.mean())
        assert torch.allclose(lse, ref_lse, atol=1e-3, rtol=0)


def test_noalloc_rejects_partials_beyond_the_array():
    pkv = _pkv()
    # 2048 single-token requests at 64 splits need far more than 8 MiB of partials
    assert pkv.pkv_workspace_bytes(2048, 32, 128, 64) > 8 << 20
    q = torch.zeros(2048, 32, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 16, 8, 128, dtype=torch.bfloat16, device="cuda")
    qsl = torch.arange(2049, dtype=torch.int32, device="cuda")
    sl = torch.ones(2048, dtype=torch.int32, device="cuda")
    bt = torch.zeros(2048, 1, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_attention_varlen_noalloc(q, kc, kc, torch.empty_like(q), qsl, sl, bt, 1, 1, 0.1,
                                         num_splits=64)
    assert e.value.code == 3                               # PKV_ERR_WORKSPACE

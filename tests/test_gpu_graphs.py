"""The CUDA-graph decode runner on the GPU against the float64 oracle: steps of
several sizes through one runner (padding to the captured size, staging slots
reused), outputs within the attention tolerance and the new tokens' cache rows
bit-exact."""

import dataclasses

import numpy as np
import pytest
import torch

import workloads
from oracle import ref
from paged_kv_attention_17_gb300 import metadata
from paged_kv_attention_17_gb300.graphs import DecodeGraphRunner
from tests.harness import to_torch

pytestmark = pytest.mark.gpu


def _subset(w, idx):
    # decode requests: request i owns token i
    return dataclasses.replace(w, requests=[w.requests[i] for i in idx], q=w.q[idx],
                               k_new=w.k_new[idx], v_new=w.v_new[idx])


@pytest.mark.parametrize("inputs", ["stage", "mapped", "memcpy"])
def test_graph_runner_steps_match_oracle(inputs):
    rng = np.random.Generator(np.random.PCG64(5))
    ctx = rng.integers(1, 700, size=8)
    w = workloads.build("graphs", "bf16", 32, 8, 128, [(int(c) - 1, 1) for c in ctx], seed=11)
    kc, vc = to_torch(w.k_pool, "bf16", "cuda"), to_torch(w.v_pool, "bf16", "cuda")
    width = 48
    runner = DecodeGraphRunner(kc, vc, 32, w.softmax_scale, width, 700, max_batch=8,
                               sizes=[1, 2, 4, 8], inputs=inputs)
    for idx in ([0], [0, 1, 2], list(range(8)), [3, 4, 5, 6, 7], [6, 2]):
        sub = _subset(w, np.array(idx))
        meta = metadata.build(sub.requests, sub.block_size)
        step = runner.begin(len(idx))
        step.q.copy_(to_torch(sub.q, "bf16", "cpu"))
        step.k_new.copy_(to_torch(sub.k_new, "bf16", "cpu"))
        step.v_new.copy_(to_torch(sub.v_new, "bf16", "cpu"))
        step.slot_mapping.copy_(torch.from_numpy(meta["slot_mapping"]))
        step.seq_lens.copy_(torch.from_numpy(meta["seq_lens"]))
        bt = meta["block_table"]
        step.block_table.zero_()
        step.block_table[:, :bt.shape[1]].copy_(torch.from_numpy(bt))
        runner.launch(step)
        out, flag = runner.result(step)
        assert flag == 0
        o_ref, _, kc_ref, vc_ref, _ = ref.paged_step(sub)
        err = np.abs(out.float().numpy().astype(np.float64) - o_ref)
        assert err.max() <= 1e-2 and err.mean() <= 1e-3, (idx, err.max(), err.mean())
        # the step's new K/V rows landed bit-exactly
        slots = meta["slot_mapping"]
        got_k = kc.view(-1, 8, 128)[torch.from_numpy(slots).cuda()].view(torch.int16).cpu().numpy()
        want_k = kc_ref.reshape(-1, 8, 128)[slots].view(np.int16)
        assert np.array_equal(got_k, want_k)


def test_graph_runner_over_an_e4m3_cache():
    rng = np.random.Generator(np.random.PCG64(6))
    ctx = rng.integers(1, 700, size=8)
    w = workloads.build("graphs_e4m3", "bf16", 32, 8, 128, [(int(c) - 1, 1) for c in ctx],
                        seed=12, kv_dtype="e4m3", k_scale=0.5, v_scale=0.25)
    kc = torch.from_numpy(w.k_pool).cuda()
    vc = torch.from_numpy(w.v_pool).cuda()
    runner = DecodeGraphRunner(kc, vc, 32, w.softmax_scale, 48, 700, max_batch=8,
                               sizes=[1, 2, 4, 8], kv_scales=(0.5, 0.25))
    for idx in ([0, 1, 2], list(range(8)), [6, 2]):
        sub = _subset(w, np.array(idx))
        meta = metadata.build(sub.requests, sub.block_size)
        step = runner.begin(len(idx))
        step.q.copy_(to_torch(sub.q, "bf16", "cpu"))
        step.k_new.copy_(to_torch(sub.k_new, "bf16", "cpu"))
        step.v_new.copy_(to_torch(sub.v_new, "bf16", "cpu"))
        step.slot_mapping.copy_(torch.from_numpy(meta["slot_mapping"]))
        step.seq_lens.copy_(torch.from_numpy(meta["seq_lens"]))
        bt = meta["block_table"]
        step.block_table.zero_()
        step.block_table[:, :bt.shape[1]].copy_(torch.from_numpy(bt))
        runner.launch(step)
        out, flag = runner.result(step)
        assert flag == 0
        o_ref, _, kc_ref, _, _ = ref.paged_step(sub)
        err = np.abs(out.float().numpy().astype(np.float64) - o_ref)
        assert err.max() <= 1e-2 and err.mean() <= 1e-3, (idx, err.max(), err.mean())
        slots = meta["slot_mapping"]
        got_k = kc.view(-1, 8, 128)[torch.from_numpy(slots).cuda()].cpu().numpy()
        assert np.array_equal(got_k, kc_ref.reshape(-1, 8, 128)[slots])


@pytest.mark.parametrize("nbytes", [16, 4096, 16 * 1000 + 16 * 7, 5 << 20])
def test_stage_inputs_copies_pinned_host_bytes_exactly(nbytes):
    import paged_kv_attention_17_gb300 as pkv
    g = torch.Generator().manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g).pin_memory()
    dst = torch.zeros(nbytes + 64, dtype=torch.uint8, device="cuda")
    pkv.pkv_stage_inputs(dst[:nbytes], src)
    dev_src = src.cuda()
    dst2 = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    pkv.pkv_stage_inputs(dst2, dev_src)            # device memory as the source too
    torch.cuda.synchronize()
    assert torch.equal(dst[:nbytes].cpu(), src)
    assert int(dst[nbytes:].count_nonzero()) == 0  # nothing written past the end
    assert torch.equal(dst2, dev_src)

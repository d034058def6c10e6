"""pkv_attention_varlen_window on the GPU against the float64 oracle.

Reading: with window W the row at position p sees keys j with p - W < j
(and the causal limit).  Same tolerances as the unwindowed path: bf16 max
|err| <= 1e-2, mean <= 1e-3; fp32 1e-4 / 1e-5.
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


def _check_lse(lse, lse_ref, tokens=None):
    got = lse.cpu().double().numpy()
    if tokens is not None:
        got, lse_ref = got[tokens], lse_ref[tokens]
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.abs(got[fin] - lse_ref[fin]).max() <= 1e-3


def _windowed(w, window):
    w.window = window
    return w


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("window", [1, 5, 16, 40, 128, 200, 1000])
@pytest.mark.parametrize("dtype,hq,hkv,d", [("bf16", 8, 2, 128), ("bf16", 4, 4, 64),
                                            ("f32", 4, 1, 128), ("bf16", 16, 1, 128)])
def test_random_small_batches(seed, window, dtype, hq, hkv, d):
    # decodes, short tails and prefill chunks (tensor-core tiles for bf16 from
    # a 128-key window on, CUDA-core tiles below)
    w = _windowed(workloads.random_small(seed + 200, dtype=dtype, hq=hq, hkv=hkv, d=d,
                                         num_seqs=6, max_new=150), window)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref, dtype)
    _check_lse(lse, lse_ref)


@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("window", [1, 17, 300])
@pytest.mark.parametrize("hq,hkv,qlen", [(32, 8, 1), (32, 8, 4), (64, 8, 1), (16, 1, 2)])
def test_decode_batches(splits, window, hq, hkv, qlen):
    rng = np.random.Generator(np.random.PCG64(hq + window + qlen))
    ctx = rng.integers(1, 900, size=9)
    shape = [(int(c), qlen) for c in ctx] + [(0, qlen), (15, qlen), (16, qlen)]
    w = workloads.build("win_decode", "bf16", hq, hkv, 128, shape, rng=rng, window=window)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev, num_splits=splits)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref, "bf16")
    _check_lse(lse, lse_ref)


def test_non_causal_window():
    w = _windowed(workloads.random_small(240, hq=8, hkv=2, d=128, causal=False), 9)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref, "bf16")
    _check_lse(lse, lse_ref)


@pytest.mark.parametrize("window", [1024, 4096])
def test_long_context_decode(window):
    # decode at context 8192: blocks below the window are skipped
    w = _windowed(workloads.decode_8k(), window)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref, "bf16")
    _check_lse(lse, lse_ref)


def test_prefill_8k_sampled_rows():
    # tensor-core prefill with a 1000-token window: rows at tile edges, the
    # window edge crossing tiles, and the last rows
    w = _windowed(workloads.prefill_8k(), 1000)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    toks = sorted({0, 1, 127, 128, 999, 1000, 1001, 1127, 1128, 2047, 2048, 4095, 5000, 8063,
                   8064, 8190, 8191})
    o_ref, lse_ref, *_ = ref.paged_step(w, tokens=toks)
    assert int(flag.item()) == 0
    _check(out, o_ref, "bf16", toks)
    _check_lse(lse, lse_ref, toks)


def test_window_zero_and_huge_equal_the_plain_call():
    w = workloads.random_small(250, hq=8, hkv=2, d=128, num_seqs=6)
    dev = device_inputs(w)
    plain, _, _ = run_step(dev, num_splits=2)
    m = dev["meta"]
    for window in (0, 1 << 20):
        out = torch.empty_like(dev["q"])
        pkv.pkv_attention_varlen(dev["q"], dev["k_cache"], dev["v_cache"], out, dev["qsl"],
                                 dev["seq_lens"], dev["block_table"], m["max_query_len"],
                                 m["max_seq_len"], w.softmax_scale, num_splits=2, window=window)
        assert torch.equal(out, plain), window

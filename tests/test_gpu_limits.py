"""Large and extreme shapes on the GPU against the float64 oracle.

A 128K-token context at the largest split count (64 splits of 128 blocks),
thousands of requests in one launch (a deep request grid), a 32K-token causal
prefill on the tensor-core path (sampled rows), and a long request on the
CUDA-core tiles (fp32, many 16-row tiles).  Tolerances as everywhere: bf16
max |err| <= 1e-2, mean <= 1e-3; fp32 1e-4 / 1e-5.
"""

import numpy as np
import pytest

import workloads
from oracle import ref
from tests.harness import device_inputs, errors, run_step

import paged_kv_attention_17_gb300 as pkv

pytestmark = pytest.mark.gpu

TOL = {"bf16": (1e-2, 1e-3), "f32": (1e-4, 1e-5)}


def _check(out, lse, w, dtype, tokens=None):
    o_ref, lse_ref, *_ = ref.paged_step(w, tokens=tokens)
    mx, mean = errors(out, o_ref, tokens)
    tmax, tmean = TOL[dtype]
    assert mx <= tmax and mean <= tmean, (mx, mean)
    got = lse.cpu().double().numpy()
    if tokens is not None:
        got, lse_ref = got[tokens], lse_ref[tokens]
    assert np.abs(got - lse_ref).max() <= 1e-3


@pytest.mark.parametrize("splits", [64, 0])
def test_decode_128k_context(splits):
    # one decode at context 131072 (8192 blocks): 64 splits of 128 blocks each
    w = workloads.build("decode_128k", "bf16", 8, 2, 128, [(131071, 1)], seed=3,
                        pool_blocks=8200)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev, num_splits=splits)
    assert int(flag.item()) == 0
    _check(out, lse, w, "bf16")


def test_thousands_of_requests():
    # 3000 decode-class requests (1-4 new tokens, contexts up to 80) in one grid
    rng = np.random.Generator(np.random.PCG64(8))
    shape = [(int(c), int(n)) for c, n in zip(rng.integers(0, 80, size=3000),
                                              rng.integers(1, 5, size=3000))]
    w = workloads.build("many", "bf16", 8, 2, 128, shape, rng=rng)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    assert int(flag.item()) == 0
    _check(out, lse, w, "bf16")


def test_prefill_32k_sampled_rows():
    w = workloads.build("prefill_32k", "bf16", 8, 2, 128, [(0, 32768)], seed=4)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    assert int(flag.item()) == 0
    toks = [0, 1, 127, 128, 4095, 16384, 20000, 32639, 32640, 32767]
    _check(out, lse, w, "bf16", toks)


def test_long_request_on_cuda_core_tiles():
    # fp32: every row of a 2500-token request on a 700-token prefix, 16-row tiles
    w = workloads.build("long_f32", "f32", 4, 1, 64, [(700, 2500), (30, 1)], seed=5)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    assert int(flag.item()) == 0
    _check(out, lse, w, "f32")


def test_split_count_bounds():
    # the automatic count never exceeds 64 nor drops below one split per 8 blocks
    for ctx in (16, 127, 128, 1024, 8192, 131072, 1 << 20):
        s = pkv.pkv_num_splits(1, 1, ctx, 32, 8, 128)
        assert 1 <= s <= 64
        assert s == 1 or s <= -(-ctx // 16) // 8

"""The E4M3 (8-bit) KV cache on the GPU against the float64 oracle.

pkv_write_e4m3 must store exactly the oracle's codes (``oracle.fp8.quantize``:
value / scale in fp32, nearest code, ties to even, saturating at 448).
pkv_attention_varlen_e4m3 is held to the bf16 bar (max |err| <= 1e-2, mean
|err| <= 1e-3): the codes widen exactly (to f16 on the tensor-core paths, to
fp32 on the CUDA-core tiles) and q rows enter the f16 contractions scaled by
powers of two (exact for every element within 2^31 of its row's largest), so
the only differences from the oracle are those of the bf16 path (fp32
accumulation, P rounded to 16 bits, bf16 output).
The sliding-window and shared-prefix forms over an E4M3 cache are held to the
same bar.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import fp8, ref
from tests.harness import device_inputs, errors, run_step

import paged_kv_attention_17_gb300 as pkv

pytestmark = pytest.mark.gpu

TMAX, TMEAN = 1e-2, 1e-3


def _check(out, o_ref, tokens=None):
    mx, mean = errors(out, o_ref, tokens)
    assert mx <= TMAX and mean <= TMEAN, (mx, mean)


def _check_lse(lse, lse_ref):
    got = lse.cpu().double().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.abs(got[fin] - lse_ref[fin]).max() <= 1e-3


# --------------------------------------------------------------------------
# The write: bit-exact codes
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("ks,vs", [(0.5, 0.25), (0.037, 1.9)])
def test_write_codes_bit_exact(dtype, ks, vs):
    w = workloads.random_small(3, dtype=dtype, hq=8, hkv=2, d=128, num_seqs=6,
                               kv_dtype="e4m3", k_scale=ks, v_scale=vs)
    dev = device_inputs(w)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_write_e4m3(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"],
                       dev["v_cache"], ks, vs, error_flag=flag)
    _, _, kc, vc, _ = ref.paged_step(w, tokens=[])
    assert int(flag.item()) == 0
    assert np.array_equal(dev["k_cache"].cpu().numpy(), kc)
    assert np.array_equal(dev["v_cache"].cpu().numpy(), vc)


def test_write_rounding_ties_saturation_and_subnormals():
    # scale 0.5 keeps x / scale exact, so midpoints between codes stay ties
    grid = fp8.decode(np.arange(0, 0x7E, dtype=np.uint8))          # 0 .. 448
    mids = (grid[:-1] + grid[1:]) / 2
    special = np.array([0.0, -0.0, 2.0 ** -10, 2.0 ** -9 * 1.5, 2.0 ** -7, 448.0, 464.0, 480.0,
                        1e4, 3e38, -1e4, -480.0])
    vals = np.concatenate([grid, mids, -mids, special]).astype(np.float32)
    hkv, d = 1, 64
    n = -(-vals.size // (hkv * d))
    x = np.zeros(n * hkv * d, dtype=np.float32)
    x[:vals.size] = vals * np.float32(0.5)
    x = x.reshape(n, hkv, d)
    k_new = torch.from_numpy(x).cuda()
    v_new = torch.from_numpy(-x).cuda()
    nb = -(-n // 16) + 1
    kc = torch.zeros(nb, 16, hkv, d, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    slots = torch.arange(n, dtype=torch.int64, device="cuda") + 16      # skip block 0
    pkv.pkv_write_e4m3(k_new, v_new, slots, kc, vc, 0.5, 0.5)
    got_k = kc.cpu().numpy().reshape(-1, hkv, d)[16:16 + n]
    got_v = vc.cpu().numpy().reshape(-1, hkv, d)[16:16 + n]
    assert np.array_equal(got_k, fp8.quantize(x, 0.5))
    assert np.array_equal(got_v, fp8.quantize(-x, 0.5))
    assert not kc.cpu().numpy()[0].any()                                 # block 0 untouched


def test_write_skips_padding_and_flags_bad_slots():
    rng = np.random.Generator(np.random.PCG64(5))
    x = torch.from_numpy(rng.standard_normal((4, 2, 64), dtype=np.float32)).cuda()
    kc = torch.full((2, 16, 2, 64), 0x11, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    slots = torch.tensor([3, -1, 40, 7], dtype=torch.int64, device="cuda")   # 40 >= 32 slots
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_write_e4m3(x, x, slots, kc, vc, 1.0, 2.0, error_flag=flag)
    assert int(flag.item()) == pkv.FLAG_BAD_SLOT
    k = kc.cpu().numpy().reshape(32, 2, 64)
    xs = x.cpu().numpy()
    assert np.array_equal(k[3], fp8.quantize(xs[0], 1.0))
    assert np.array_equal(k[7], fp8.quantize(xs[3], 1.0))
    untouched = [s for s in range(32) if s not in (3, 7)]
    assert (k[untouched] == 0x11).all()


# --------------------------------------------------------------------------
# Attention over the codes
# --------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 128), (4, 4, 64), (32, 4, 128), (16, 1, 128),
                                      (16, 1, 64)])
def test_random_small_batches(seed, hq, hkv, d):
    # decodes, short tails (register-q tiles) and prefill chunks (CUDA-core tiles)
    w = workloads.random_small(seed + 100, hq=hq, hkv=hkv, d=d, num_seqs=6, kv_dtype="e4m3",
                               k_scale=0.5, v_scale=0.25)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref)
    _check_lse(lse, lse_ref)


@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("hq,hkv,d,qlen", [(32, 8, 128, 1), (32, 8, 128, 3), (16, 2, 64, 1),
                                           (64, 8, 128, 1), (8, 8, 128, 4)])
def test_decode_batches_split_and_unsplit(splits, hq, hkv, d, qlen):
    rng = np.random.Generator(np.random.PCG64(hq * 7 + qlen))
    ctx = rng.integers(1, 700, size=9)
    shape = [(int(c), qlen) for c in ctx] + [(0, qlen), (15, qlen), (16, qlen)]
    w = workloads.build("fp8_decode", "bf16", hq, hkv, d, shape, rng=rng, kv_dtype="e4m3",
                        k_scale=0.7, v_scale=0.3)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev, num_splits=splits)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref)
    _check_lse(lse, lse_ref)


def test_non_causal():
    w = workloads.random_small(140, hq=8, hkv=2, d=128, causal=False, kv_dtype="e4m3",
                               k_scale=0.5, v_scale=0.5)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref)
    _check_lse(lse, lse_ref)


def test_decode_8k_full_size_bench_configuration():
    # the automatic split count, as the benchmark runs it; every output row
    w = workloads.decode_8k_e4m3()
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref)
    _check_lse(lse, lse_ref)


def test_batched_decode_64_full_size():
    w = workloads.batched_decode_64_e4m3()
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref)
    _check_lse(lse, lse_ref)


def test_matches_the_bf16_path_on_the_dequantised_cache():
    # the same step through the bf16 kernels on a cache holding scale * value
    # (exact in bf16: 4 significant bits times a power of two).  Decode rows
    # run the same fp32 arithmetic on both paths, so they agree to one bf16
    # rounding (|out| < 1 here: 2^-8); prefill rows of the bf16 path take the
    # tensor-core kernel, whose bf16 P differs more and is held to the oracle
    # bar by the other tests.
    w = workloads.random_small(150, hq=8, hkv=2, d=128, num_seqs=8, kv_dtype="e4m3",
                               k_scale=0.5, v_scale=0.25)
    dev = device_inputs(w)
    out8, _, _ = run_step(dev)
    kc = (0.5 * fp8.decode(dev["k_cache"].cpu().numpy())).astype(np.float32)
    vc = (0.25 * fp8.decode(dev["v_cache"].cpu().numpy())).astype(np.float32)
    kb = torch.from_numpy(kc).to(torch.bfloat16).cuda()
    vb = torch.from_numpy(vc).to(torch.bfloat16).cuda()
    out16 = torch.empty_like(dev["q"])
    m = dev["meta"]
    pkv.pkv_attention_varlen(dev["q"], kb, vb, out16, dev["qsl"], dev["seq_lens"],
                             dev["block_table"], m["max_query_len"], m["max_seq_len"],
                             w.softmax_scale, causal=w.causal)
    qsl = m["query_start_loc"]
    rows = [t for r in range(len(qsl) - 1) if qsl[r + 1] - qsl[r] <= pkv.PKV_DECODE_MAX_QLEN
            for t in range(qsl[r], qsl[r + 1])]
    assert rows
    diff = (out8.float() - out16.float())[rows].abs().max().item()
    assert diff <= 2.0 ** -8, diff


# --------------------------------------------------------------------------
# Requests longer than the decode bound at head_dim 128: the tcgen05 prefill
# tiles, over codes widened to f16 in shared memory and q rows rescaled to f16
# --------------------------------------------------------------------------

@pytest.mark.parametrize("hq,hkv", [(8, 2), (32, 8), (4, 4), (12, 4)])
@pytest.mark.parametrize("causal", [True, False])
def test_tensor_core_prefill(hq, hkv, causal):
    # head pairs (even groups) and tile pairs (groups 1 and 3); 1, 2, 3 and 9
    # query tiles with ragged tails, on empty and cached prefixes, beside
    # decode rows and short tails
    shape = [(0, 100), (300, 256), (40, 300), (1000, 1), (0, 1100), (77, 5)]
    w = workloads.build("fp8_prefill", "bf16", hq, hkv, 128, shape, seed=hq * 5 + hkv,
                        causal=causal, kv_dtype="e4m3", k_scale=0.45, v_scale=0.3)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref)
    _check_lse(lse, lse_ref)


@pytest.mark.parametrize("window", [0, 300])
def test_tensor_core_prefill_long_chunk(window):
    # a 2048-token chunk on a 1000-token prefix at GQA 32/8, every row
    w = workloads.build("fp8_chunk", "bf16", 32, 8, 128, [(1000, 2048), (300, 1)], seed=81,
                        window=window, kv_dtype="e4m3", k_scale=0.5, v_scale=0.5)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref)
    _check_lse(lse, lse_ref)


def test_tensor_core_prefill_q_rows_of_any_magnitude():
    # every (token, head) row of q scaled by its own power of two in
    # 2^-8 .. 2^20 (exact in bf16), with softmax_scale 2^-14 / sqrt(D) keeping
    # the largest rows' scores moderate: rows up to ~5e6 in magnitude, beyond
    # f16's 65504, are rewritten as f16 scaled to their own range, beside rows
    # so small their softmax is near uniform
    w = workloads.build("fp8_qscale", "bf16", 8, 2, 128, [(0, 300), (50, 130), (200, 1)],
                        seed=91, kv_dtype="e4m3", k_scale=0.5, v_scale=0.5,
                        scale=2.0 ** -14 / np.sqrt(128))
    rng = np.random.Generator(np.random.PCG64(92))
    f = np.ldexp(1.0, rng.integers(-8, 21, size=w.q.shape[:2]))[..., None]
    q = (w.q.astype(np.uint32) << 16).view(np.float32) * f.astype(np.float32)
    w.q = workloads.f32_to_bf16_bits(q)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref)
    _check_lse(lse, lse_ref)


def test_tensor_core_prefill_ignores_codes_past_the_context():
    # every slot no request reads holds the NaN code 0x7F: the key rows of a
    # last tile past the context are zeroed when widened, so nothing leaks
    w = workloads.build("fp8_stale", "bf16", 8, 2, 128, [(0, 200), (30, 150), (500, 1)],
                        seed=93, kv_dtype="e4m3", k_scale=0.5, v_scale=0.5, pool_blocks=64)
    dev = device_inputs(w)
    meta = dev["meta"]
    used = np.zeros(w.num_blocks * 16, dtype=bool)
    for r, L in enumerate(meta["seq_lens"]):
        for j in range(int(L)):
            used[int(meta["block_table"][r, j // 16]) * 16 + j % 16] = True
    stale = torch.from_numpy(~used).cuda()
    for c in (dev["k_cache"], dev["v_cache"]):
        c.view(w.num_blocks * 16, -1)[stale] = 0x7F
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    assert torch.isfinite(out.float()).all()
    _check(out, o_ref)
    _check_lse(lse, lse_ref)


def test_prefill_8k_full_size_all_rows():
    # all 8192 rows x 32 heads of the 8k causal prefill over an E4M3 cache
    w = workloads.prefill_8k_e4m3()
    dev = device_inputs(w)
    out, lse, flag = run_step(dev)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    _check(out, o_ref)
    _check_lse(lse, lse_ref)


@pytest.mark.parametrize("window", [1, 16, 100, 1000])
@pytest.mark.parametrize("splits", [0, 3])
def test_sliding_window_over_e4m3_cache(window, splits):
    # pkv_attention_varlen_e4m3_window: decodes, short tails and prefill
    # chunks, each row keeping only its `window` most recent keys
    rng = np.random.Generator(np.random.PCG64(window * 13 + splits))
    ctx = rng.integers(1, 1500, size=8)
    shape = [(int(c), 1) for c in ctx] + [(200, 3), (0, 40), (900, 130), (16, 1)]
    w = workloads.build("fp8_window", "bf16", 32, 8, 128, shape, rng=rng, kv_dtype="e4m3",
                        k_scale=0.6, v_scale=0.4, window=window)
    dev = device_inputs(w)
    out, lse, flag = run_step(dev, num_splits=splits)
    o_ref, lse_ref, *_ = ref.paged_step(w)
    assert int(flag.item()) == 0
    if window == 1:
        # one visible key: each output is that key's dequantised V, a value
        # bf16 cannot hold, so the bound is bf16's own rounding of it (the
        # absolute bounds assume averaged outputs; these reach |o| ~ 5)
        got = out.float().cpu().double().numpy()
        assert np.all(np.abs(got - o_ref) <= 2.0 ** -8 * np.abs(o_ref) + 1e-30)
    else:
        _check(out, o_ref)
    _check_lse(lse, lse_ref)


def test_window_zero_over_e4m3_is_the_plain_call():
    w = workloads.build("fp8_w0", "bf16", 16, 4, 128, [(300, 1), (40, 5), (1000, 1)], seed=3,
                        kv_dtype="e4m3", k_scale=0.5, v_scale=0.5)
    dev = device_inputs(w)
    out0, lse0, flag0 = run_step(dev, num_splits=2)
    m = dev["meta"]
    out1 = torch.empty_like(out0)
    pkv.pkv_attention_varlen_e4m3(dev["q"], dev["k_cache"], dev["v_cache"], out1, dev["qsl"],
                                  dev["seq_lens"], dev["block_table"], m["max_query_len"],
                                  m["max_seq_len"], w.softmax_scale, w.k_scale, w.v_scale,
                                  num_splits=2, window=0)
    huge = torch.empty_like(out0)
    pkv.pkv_attention_varlen_e4m3(dev["q"], dev["k_cache"], dev["v_cache"], huge, dev["qsl"],
                                  dev["seq_lens"], dev["block_table"], m["max_query_len"],
                                  m["max_seq_len"], w.softmax_scale, w.k_scale, w.v_scale,
                                  num_splits=2, window=1 << 20)
    torch.cuda.synchronize()
    assert int(flag0.item()) == 0
    assert torch.equal(out0, out1) and torch.equal(out0, huge)

"""Pins of the oracle's E4M3 codec (oracle/fp8.py): PyTorch's float8_e4m3fn
conversion (a library routine) inside the finite range, closed forms of the
format, and the round trip over every code."""

import numpy as np
import torch

from oracle import fp8


def _torch_codes(x32):
    return torch.from_numpy(x32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_matches_torch_inside_finite_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)
    ] + [np.linspace(-464, 464, 4001), rng.uniform(-2 ** -6, 2 ** -6, 5000)]).astype(np.float32)
    x = x[np.abs(x) < 464]                      # beyond, torch gives NaN and the format saturates
    x = x[x != 0]
    assert np.array_equal(fp8.encode(x.astype(np.float64)), _torch_codes(x))


def test_ties_go_to_the_even_mantissa():
    # every finite code but negative zero (it would pair with +0 as equals)
    grid = np.array([c for c in range(256) if (c & 0x7F) != 0x7F and c != 0x80], dtype=np.uint8)
    vals = fp8.decode(grid)
    order = np.argsort(vals)
    v, c = vals[order], grid[order]
    pos = (v[:-1] >= 0) & (v[1:] > 0)
    mids = ((v[:-1] + v[1:]) / 2)[pos]
    want = np.where((c[:-1][pos] & 1) == 0, c[:-1][pos], c[1:][pos])
    assert np.array_equal(fp8.encode(mids), want)
    assert np.array_equal(_torch_codes(mids.astype(np.float32)), want)


def test_closed_forms():
    cases = {1.0: 0x38, -2.0: 0xC0, 0.5: 0x30, 448.0: 0x7E, -448.0: 0xFE, 1.75: 0x3E,
             2.0 ** -6: 0x08, 2.0 ** -9: 0x01, 7 * 2.0 ** -9: 0x07,
             2.0 ** -10: 0x00,                   # halfway between 0 and 2^-9: even (0)
             3 * 2.0 ** -10: 0x02,               # halfway between 1 and 2 (x 2^-9): even (2)
             460.0: 0x7E, 1000.0: 0x7E, -1e6: 0xFE, 1e30: 0x7E}   # saturation
    for v, c in cases.items():
        assert int(fp8.encode(np.array([v]))[0]) == c, (v, c)
    assert int(fp8.encode(np.array([np.nan]))[0]) == 0x7F
    # the format has no infinity: +-inf saturate like any magnitude past 448
    assert fp8.encode(np.array([np.inf, -np.inf])).tolist() == [0x7E, 0xFE]
    assert fp8.quantize(np.array([np.inf, -np.inf], dtype=np.float32), 0.5).tolist() == [0x7E, 0xFE]
    assert fp8.decode([0x7E])[0] == 448.0 and fp8.decode([0x01])[0] == 2.0 ** -9
    assert np.isnan(fp8.decode([0x7F, 0xFF])).all()


def test_every_code_round_trips():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(fp8.encode(fp8.decode(codes)), codes)
    # monotone: the positive codes increase with the code
    pos = fp8.decode(np.arange(0, 0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)


def test_quantize_divides_in_float32():
    x = np.array([1.0, 3.0, 0.1, -7.25], dtype=np.float32)
    s = 0.3
    want = fp8.encode((x / np.float32(s)).astype(np.float32).astype(np.float64))
    assert np.array_equal(fp8.quantize(x, s), want)


# --------------------------------------------------------------------------
# Attention over an E4M3 cache (oracle.ref with kv_dtype="e4m3")
# --------------------------------------------------------------------------

import dataclasses  # noqa: E402

import workloads  # noqa: E402
from oracle import ref  # noqa: E402


def _fp8_workload(seed, shape, hq=8, hkv=2, d=64, ks=0.5, vs=0.25):
    return workloads.build("fp8", "bf16", hq, hkv, d, shape, seed=seed, kv_dtype="e4m3",
                           k_scale=ks, v_scale=vs)


def test_fp8_equals_fp32_on_the_dequantised_cache():
    # the scales act as K = k_scale * value, V = v_scale * value: the same
    # step on float32 caches holding those values gives the same result
    w = _fp8_workload(7, [(40, 3), (17, 1), (0, 5)])
    o, lse, kc, vc, meta = ref.paged_step(w)
    kf = (w.k_scale * fp8.decode(kc)).astype(np.float32)
    vf = (w.v_scale * fp8.decode(vc)).astype(np.float32)
    o2, lse2 = ref.attention(ref.upcast(w.q, "bf16").astype(np.float32), kf, vf,
                             meta["query_start_loc"], meta["seq_lens"], meta["block_table"],
                             num_q_heads=8, num_kv_heads=2, softmax_scale=w.softmax_scale,
                             dtype="f32")
    assert np.abs(o - o2).max() < 1e-12 and np.abs(lse - lse2).max() < 1e-12


def test_fp8_single_key_is_the_written_v():
    w = _fp8_workload(8, [(0, 1), (0, 1)], ks=0.3, vs=0.7)
    o, _, _, _, _ = ref.paged_step(w)
    v = ref.upcast(w.v_new, "bf16").astype(np.float32)             # [2, hkv, d]
    want = 0.7 * fp8.decode(fp8.quantize(v, 0.7))
    for t in range(2):
        for h in range(8):
            assert np.array_equal(o[t, h], want[t, h // 4])


def test_fp8_zero_query_gives_the_mean_of_visible_v():
    w = _fp8_workload(9, [(20, 1)], hq=4, hkv=1, vs=0.5)
    w = dataclasses.replace(w, q=np.zeros_like(w.q))
    o, _, _, vc, meta = ref.paged_step(w)
    V = 0.5 * fp8.decode(ref.gather(vc, meta["block_table"][0], 21, 16))
    assert np.abs(o[0, 0] - V[:, 0, :].mean(0)).max() < 1e-12


def _decode_pin_holds():
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().double().numpy()
    got = fp8.decode(codes)
    return bool(np.array_equal(np.isnan(got), np.isnan(want)) and
                np.array_equal(got[~np.isnan(got)], want[~np.isnan(want)]))


def test_decode_matches_torch_for_every_code():
    assert _decode_pin_holds()


def test_planted_exponent_bias_is_caught(monkeypatch):
    orig = fp8.decode
    monkeypatch.setattr(fp8, "decode", lambda c: orig(c) / 2.0)      # bias 8 instead of 7
    assert not _decode_pin_holds()


def test_planted_subnormal_scale_is_caught(monkeypatch):
    orig = fp8.decode

    def wrong(c):
        c = np.asarray(c, dtype=np.uint8)
        v = orig(c)
        sub = ((c >> 3) & 0xF) == 0
        return np.where(sub, v * 2.0, v)                                # m/8 * 2^-5
    monkeypatch.setattr(fp8, "decode", wrong)
    assert not _decode_pin_holds()

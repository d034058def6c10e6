"""The two-term E4M3 split of q rows that the E4M3 decode contraction uses.

Over an E4M3 cache the decode kernel scales each bf16 q row by a power of two
into [2^7, 2^8) and writes every element x as hi + lo: hi = x rounded to E4M3,
lo = (x - hi) rounded to E4M3, so that K's codes enter E4M3 MMAs as they are.
The remainder keeps x's last bit, which must lie on E4M3's 2^-9 grid for the
sum to be exact.  This checks, for every positive bf16 value below 2^8 and
with E4M3 rounding as the oracle's pinned encoder defines it: hi + lo == x
exactly for x >= 2^-2 (every element within 2^9 of a row maximum of at least
2^7), and |hi + lo - x| <= 2^-10 below (at most 2^-17 of that maximum).
"""
import numpy as np

from oracle import fp8


def _split(x):
    hi = fp8.decode(fp8.quantize(x.astype(np.float32), 1.0)).astype(np.float64)
    lo = fp8.decode(fp8.quantize((x - hi).astype(np.float32), 1.0)).astype(np.float64)
    return hi, lo


def _bf16_values(lo, hi):
    bits = np.arange(0x0000, 0x7F80, dtype=np.uint32)
    x = (bits << 16).view(np.float32).astype(np.float64)
    return x[(x >= lo) & (x < hi)]


def test_split_is_exact_from_a_quarter_up():
    x = _bf16_values(2.0 ** -2, 2.0 ** 8)
    hi, lo = _split(x)
    assert np.array_equal(hi + lo, x)
    xn = -x                                   # the sign carries through both terms
    hi, lo = _split(xn)
    assert np.array_equal(hi + lo, xn)


def test_split_error_below_a_quarter_is_at_most_2_to_minus_10():
    x = _bf16_values(2.0 ** -40, 2.0 ** -2)
    hi, lo = _split(x)
    err = np.abs(hi + lo - x)
    assert err.max() <= 2.0 ** -10
    assert err.max() > 0                      # the bound is reached: not exact there


def test_row_maximum_range_keeps_hi_finite():
    # the row maximum lands in [2^7, 2^8): below E4M3's 448, so hi never saturates
    x = _bf16_values(2.0 ** 7, 2.0 ** 8)
    hi, lo = _split(x)
    assert np.all(np.abs(hi) <= 448.0) and np.array_equal(hi + lo, x)

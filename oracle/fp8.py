"""FP8 E4M3 codes for an 8-bit KV cache (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The pages name an FP8 KV cache as a backend feature ("Model execution",
section "Where it breaks": not all backends support FP8 KV cache; "Anatomy of
a serving engine", exercise on the KV arithmetic with an FP8 cache) but fix no
format.  The reading taken: E4M3 codes - 1 sign bit, 4 exponent bits with bias
7, 3 mantissa bits; exponent field 0 holds subnormals m/8 * 2^-6; the largest
finite magnitude is 1.75 * 2^8 = 448; there are no infinities and the codes
S.1111.111 are NaN - with one fp32 scale per cache tensor: a cached element
stands for scale * value(code).  Encoding rounds to the nearest code, ties to
the even mantissa, and saturates magnitudes beyond 448 to 448; infinities
saturate the same way (the format has none).

Written from that definition with exact float64 arithmetic; pinned in
``tests/test_oracle_fp8.py`` against PyTorch's float8_e4m3fn conversion
(inside the finite range) and closed forms.
"""

from __future__ import annotations

import numpy as np

MAX_FINITE = 448.0
NAN_CODE = 0x7F


def decode(codes) -> np.ndarray:
    """float64 value of each E4M3 code (NaN for the NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def encode(x) -> np.ndarray:
    """Nearest E4M3 code of each value (ties to even, saturating at 448, +-inf
    included; NaN to the NaN code).  Values are exact float64 (e.g. float32
    inputs)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint8)
    flat, res = x.ravel(), out.ravel()
    for k, v in enumerate(flat):
        if np.isnan(v):
            res[k] = NAN_CODE
            continue
        s = 0x80 if np.signbit(v) else 0
        a = abs(v)
        if np.isinf(a):                           # no infinities in E4M3: saturate
            res[k] = s | 0x7E
        elif a >= 2.0 ** -6:                      # normal range
            mant, e = np.frexp(a)                 # a = mant * 2^e, mant in [0.5, 1)
            e -= 1                                # a = (2 mant) * 2^e, 2 mant in [1, 2)
            q = np.round((2.0 * mant - 1.0) * 8.0)   # ties to even
            if q == 8.0:
                q, e = 0.0, e + 1
            if e > 8 or (e == 8 and q > 6.0):      # beyond 448: saturate
                res[k] = s | 0x7E
            else:
                res[k] = s | ((e + 7) << 3) | int(q)
        else:                                     # subnormal range (may round up to 2^-6)
            q = int(np.round(a / 2.0 ** -9))      # ties to even; q == 8 is the code 0x08
            res[k] = s | q
    return out


def quantize(x_f32, scale: float) -> np.ndarray:
    """Codes of x / scale, the division taken in float32 (round to nearest)."""
    xs = (np.asarray(x_f32, dtype=np.float32) / np.float32(scale)).astype(np.float32)
    return encode(xs.astype(np.float64))

"""The FP4 activation encoder's exponent rule, checked on the CPU.

The GPU encoder takes the block exponent k = ceil(log2(fl(amax / 6))) (the
ceiling of log2 of the quotient rounded once to float32, ds4.c FP4 activation
quantisation) without dividing: amax = m * 2^e (m in [1, 2), 8 significant
bits for a bf16 amax) gives k = e - 2 + (m > 1.5), with amax floored at
6 * 2^-126 and k = 127 for an infinite amax.  That identity is what this test
checks, for every bf16 magnitude, against the quotient computed in float32 and
its ceiling taken exactly with frexp.
"""
import math

import numpy as np


def _ceil_log2_exact(q: float) -> int:
    m, ex = math.frexp(q)          # q = m * 2^ex, m in [0.5, 1)
    return ex - 1 if m == 0.5 else ex


def test_division_free_exponent_matches_float32_quotient_for_every_bf16_amax():
    mags = np.arange(0, 0x7F81, dtype=np.uint32)                 # +0 .. +inf, NaN excluded
    amax = (mags << 16).view(np.float32)
    amax = np.maximum(amax, np.float32(6.0 * 2.0 ** -126))
    with np.errstate(over="ignore"):
        q = (amax / np.float32(6.0)).astype(np.float32)
    want = np.array([127 if math.isinf(v) else _ceil_log2_exact(float(v)) for v in q])
    ab = np.maximum(mags, 0x01C0)                                 # 0x01C0 = 1.5 * 2^-124
    got = np.where(ab >= 0x7F80, 127, (ab >> 7).astype(np.int64) - 129 + ((ab & 0x7F) > 0x40))
    np.testing.assert_array_equal(got, want)
    assert want.min() == -126 and want.max() == 127

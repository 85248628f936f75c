"""The store kernel computes amax / 6 without a division instruction:
q0 = amax * RN(1/6), r = fma(-q0, 6, amax), q = fma(r, RN(1/6), q0)
(Markstein's quotient correction with an exact FMA residual).  This test
checks, in exact rational arithmetic, that the sequence equals the IEEE
fp32 quotient for every finite non-negative bf16 and fp16 value -- the only
values amax can take -- and that the residual is always exact.  CPU
only."""
from fractions import Fraction as F

import numpy as np

INV6 = np.uint32(0x3E2AAAAB).view(np.float32)


def rn32(x: F) -> np.float32:
    """Round a rational to the nearest fp32, ties to even (subnormals
    included)."""
    if x == 0:
        return np.float32(0.0)
    c = np.float32(float(x))
    cands = [np.nextafter(c, np.float32(-np.inf)), c,
             np.nextafter(c, np.float32(np.inf))]
    return min(cands, key=lambda v: (abs(F(float(v)) - x),
                                     int(np.float32(v).view(np.uint32)) & 1))


def test_inv6_constant():
    assert INV6 == np.float32(1.0) / np.float32(6.0)


def _check_all(a):
    ieee = a / np.float32(6.0)
    q0 = a * INV6  # fp32 products, correctly rounded
    c = F(float(INV6))
    for i in range(a.size):
        x, q = F(float(a[i])), F(float(q0[i]))
        res = x - 6 * q
        r = rn32(res)
        assert F(float(r)) == res, a[i]          # fma residual is exact
        q1 = rn32(F(float(r)) * c + q)            # one rounding, as fma
        assert q1 == ieee[i], (a[i], q1, ieee[i])


def test_fma_corrected_division_by_six_is_exact_for_all_bf16():
    bits = np.arange(0, 0x7F80, dtype=np.uint32)  # finite, non-negative
    _check_all((bits << 16).view(np.float32))


def test_fma_corrected_division_by_six_is_exact_for_all_fp16():
    bits = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16)
    _check_all(bits.view(np.float16).astype(np.float32))

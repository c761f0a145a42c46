"""The append's block-scale quotient RN32(amax / d) from a precomputed reciprocal (CPU only).

The kernels compute the candidate scale ratio amax / RN32(k * gs) without a division: with
rb = RN32(1 / b),
    q0 = RN32(a * rb),   r = RN32(a - q0 * b) (fused),   q = RN32(q0 + r * rb) (fused),
which is Markstein's correctly rounded division for normal operands and quotients
(P. Markstein, "IA-64 and Elementary Functions", 2000, the division theorem). This test
emulates that sequence exactly and compares it with IEEE binary32 division (numpy's float32
divide, correctly rounded), for every positive finite fp16 and bf16 value of the block
amax against a seeded sample of divisors:
  * products of two binary32 values are exact in binary64;
  * a - q0*b is exact in binary64 (Sterbenz: q0*b is within a factor of two of a), so its
    one rounding to binary32 is numpy's float32 conversion;
  * q0 + r*rb is rounded to binary64 first; that second rounding can only change the final
    binary32 result when the binary64 value lands exactly on a binary32 midpoint, and those
    cases are recomputed in exact rational arithmetic.
The kernels rely on the sequence for normal b and rb (otherwise they divide). The result
must equal IEEE division wherever the quotient lies in [2^-12, 2^20); outside it, the
block scale is E4M3(fminf(q, cap)) with q below E4M3's smallest rounding threshold
(2^-10) or above any cap, so it only has to land on the same side, which is checked too
(where the quotient overflows, the sequence gives NaN and fminf takes the cap).
"""
from fractions import Fraction

import pytest

import numpy as np
import torch

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

LO, HI = 2.0 ** -12, 2.0 ** 20


def amax_values() -> np.ndarray:
    """Every positive finite fp16 and bf16 value, as binary32."""
    h = np.arange(1, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float32)
    b = torch.from_numpy(np.arange(1, 0x7F80, dtype=np.int32).astype(np.int16)).view(
        torch.bfloat16).float().numpy()
    return np.unique(np.concatenate([h, b]))


def divisors(n: int = 1500, seed: int = 77) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    m = rng.integers(1 << 23, 1 << 24, n).astype(np.float64)
    e = rng.integers(-60, 60, n)
    b = np.ldexp(m, e - 23).astype(np.float32)
    gs = np.ldexp(rng.uniform(1, 2, n // 3), rng.integers(-40, 20, n // 3)).astype(np.float32)
    special = np.array([1.0, 1.5, 2.0 ** -20, 3.0 * 2.0 ** 7, 6.0 * 2.0 ** -10, 1.0 + 2.0 ** -23,
                        2.0 - 2.0 ** -23], np.float32)
    out = np.concatenate([b, (np.float32(6) * gs).astype(np.float32),
                          (np.float32(4) * gs).astype(np.float32), special])
    rb = (np.float32(1) / out).astype(np.float32)
    tiny, big = np.finfo(np.float32).tiny, np.finfo(np.float32).max
    keep = (out >= tiny) & (out <= big) & (rb >= tiny) & (rb <= big)
    return out[keep]


def rn32_exact(q: Fraction) -> np.float32:
    """q (a positive normal-range rational) rounded to binary32, ties to even."""
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    elif Fraction(2) ** (e + 1) <= q:
        e += 1
    spacing = Fraction(2) ** (e - 23)
    return np.float32(float(round(q / spacing) * spacing))


def markstein(a: np.ndarray, b: np.float32):
    rb = np.float32(1) / b
    q0 = (a * rb).astype(np.float32)
    p = q0.astype(np.float64) * np.float64(b)                  # exact
    r = (a.astype(np.float64) - p).astype(np.float32)          # exact difference, one rounding
    y = q0.astype(np.float64) + r.astype(np.float64) * np.float64(rb)  # rounded to binary64
    q = y.astype(np.float32)
    # binary32 midpoints in binary64: the 29 bits below binary32 precision are 1000...0
    low = y.view(np.uint64) & np.uint64((1 << 29) - 1)
    mid = np.nonzero((low == np.uint64(1 << 28)) & (y >= LO / 2) & (y < HI * 2))[0]
    for i in mid:
        exact = Fraction(float(q0[i])) + Fraction(float(r[i])) * Fraction(float(rb))
        q[i] = rn32_exact(exact)
    return q, len(mid)


def test_reciprocal_division_matches_ieee():
    a = amax_values()
    assert a.size > 60000
    mids = checked = 0
    for b in divisors():
        q, nm = markstein(a, b)
        mids += nm
        ieee = (a / b).astype(np.float32)
        exact_q = a.astype(np.float64) / np.float64(b)
        inside = (exact_q >= LO) & (exact_q < HI)
        bad = np.nonzero(inside & (q != ieee))[0]
        assert bad.size == 0, (float(b), a[bad[:5]], q[bad[:5]], ieee[bad[:5]])
        checked += int(inside.sum())
        # outside the range: below 2^-10 (E4M3's lowest threshold), or clamped to any cap by
        # the kernels' fminf, which also takes the cap when the sequence overflows to NaN
        below, above = exact_q < LO, exact_q >= HI
        assert np.all(q[below] < 2.0 ** -10) and np.all(q[below] >= 0), float(b)
        assert np.all(np.fmin(q[above], np.float32(448)) == 448), float(b)
    assert checked > 20_000_000, checked

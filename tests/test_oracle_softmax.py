"""Pins for the oracle's fp32 exponential, pairwise sum and softmax.

The fp32 softmax is the routing decision chain's arithmetic; these tests tie
it to mathematics (exact rationals, exp in double, exact sums), not to itself.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import moe_oracle as O


def _ulp32(v: np.ndarray) -> np.ndarray:
    v = np.abs(np.asarray(v, dtype=np.float64)).astype(np.float32)
    return np.spacing(v).astype(np.float64)


def test_taylor_coefficients_are_correctly_rounded():
    for k, c in enumerate(O.TAYLOR):
        exact = Fraction(1, math.factorial(k))
        c = np.float32(c)
        lo = np.nextafter(c, np.float32(0))
        hi = np.nextafter(c, np.float32(1))
        err = abs(Fraction(float(c)) - exact)
        assert err <= abs(Fraction(float(lo)) - exact)
        assert err <= abs(Fraction(float(hi)) - exact)


def test_cody_waite_split():
    # LN2_HI has 9 significant bits, so n * LN2_HI is exact for the exponents used.
    for n in range(-130, 1):
        prod = np.float32(n) * O.LN2_HI
        assert Fraction(float(prod)) == n * Fraction(float(O.LN2_HI))
    # HI + LO approximates ln 2 to well below fp32 resolution.
    assert abs(float(O.LN2_HI) + float(O.LN2_LO) - math.log(2.0)) < 1e-11


def test_exp_within_two_ulp_of_double_exp():
    rng = np.random.default_rng(1)
    u = np.concatenate([
        np.linspace(-86.9, 0.0, 2_000_001, dtype=np.float32),
        (-rng.random(500_000) * 20).astype(np.float32),
        (-rng.random(500_000) * 1e-3).astype(np.float32),
    ])
    got = O.exp_f32(u).astype(np.float64)
    ref = np.exp(u.astype(np.float64))
    ulps = np.abs(got - ref) / _ulp32(ref)
    assert ulps.max() <= 2.0, ulps.max()


def test_exp_special_values():
    assert O.exp_f32(np.float32(0.0)) == np.float32(1.0)
    assert O.exp_f32(np.float32(-100.0)) == 0.0
    # n = rint(u*log2e) < -125 flushes to 0 (the result would leave the normal range)
    assert O.exp_f32(np.float32(-87.5)) == 0.0
    assert O.exp_f32(np.float32(-86.9)) > 0.0
    # arguments near the range-reduction boundaries (u close to -k ln 2 and
    # -(k + 1/2) ln 2): within 2 ulp of exp of the same fp32 argument
    for k in range(0, 125):
        for off in (0.0, 0.5):
            u0 = np.float32(-(k + off) * math.log(2.0))
            for u in (np.nextafter(u0, np.float32(-1e9)), u0, np.nextafter(u0, np.float32(0))):
                if u > 0:
                    continue
                ref = math.exp(float(u))
                v = float(O.exp_f32(np.float32(u)))
                assert abs(v - ref) <= 2 * float(np.spacing(np.float32(ref))), (k, off, u)


def test_pairwise_sum_order():
    # Stride-halving order (v[i] += v[i+h]) differs from left-to-right here:
    # pairwise gives 1 + 2^-23, sequential gives 1 (ties to even).
    q = np.array([1.0, 2.0**-24, 0.0, 2.0**-24], dtype=np.float32)
    assert O.pairwise_sum_f32(q) == np.float32(1.0 + 2.0**-23)
    seq = np.float32(0)
    for v in q:
        seq = np.float32(seq + v)
    assert seq == np.float32(1.0)


def test_pairwise_sum_accuracy_and_padding():
    rng = np.random.default_rng(2)
    for E in (1, 3, 4, 5, 8, 33, 64):
        q = rng.random((200, E)).astype(np.float32)
        s = O.pairwise_sum_f32(q).astype(np.float64)
        exact = np.array([math.fsum(map(float, row)) for row in q])
        assert np.all(np.abs(s - exact) <= E * _ulp32(exact))
        # small integers sum exactly in any order
        qi = rng.integers(0, 100, (50, E)).astype(np.float32)
        assert np.array_equal(O.pairwise_sum_f32(qi), qi.sum(axis=1, dtype=np.float64).astype(np.float32))


@pytest.mark.parametrize("E", [4, 8, 64])
def test_softmax_close_to_exact_and_normalised(E):
    rng = np.random.default_rng(E)
    l = (rng.standard_normal((4000, E)) * 3).astype(np.float32)
    p = O.softmax_f32(l).astype(np.float64)
    ref = O.softmax_f64(l.astype(np.float64))
    # error bound vs the exact softmax of the same fp32 logits: exp (2 ulp),
    # the sum (E ulp), the division (1/2 ulp), plus the rounding of u = l - m,
    # which moves e^u by a relative |u| 2^-24
    u = np.abs(l.astype(np.float64) - l.max(axis=1, keepdims=True))
    bound = ref * ((3.0 + E) * 2.0**-23 + u * 2.0**-24)
    err = np.abs(p - ref)
    assert np.all(err <= bound), (err / bound).max()
    assert np.all(np.abs(p.sum(axis=1) - 1.0) <= E * 2.0**-23)
    # the largest logit gets the largest probability
    assert np.array_equal(np.argmax(p, axis=1), np.argmax(l, axis=1))


def test_softmax_bits_invariant_under_a_shift_of_the_logits():
    """softmax(l + c) = softmax(l). With logits on a 2^-10 grid and |l| < 32,
    l + c is exact in fp32 for c = 96 and c = 1000, and so is l + c - max; the
    specified arithmetic (subtract the row maximum first) therefore gives the
    same bits. Without the max subtraction e^(l + c) leaves the fp32 range."""
    rng = np.random.default_rng(5)
    l = np.clip(np.round(rng.standard_normal((2000, 8)) * 3 * 1024) / 1024, -31, 31)
    l = l.astype(np.float32)
    p = O.softmax_f32(l)
    for c in (96.0, 1000.0):
        lc = (l + np.float32(c)).astype(np.float32)
        assert np.array_equal(lc.astype(np.float64) - c, l.astype(np.float64))   # exact shift
        assert np.array_equal(O.softmax_f32(lc).view(np.uint32), p.view(np.uint32))

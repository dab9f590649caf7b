"""The tolerance of the inv_rms parity tests, checked at the extremes.

The GPU kernels evaluate the power mean of a row's block scales as
  m = max_k e_k,
  S = sum_k [t_k >= 0] 2^t_k,  t_k = 48 + p (e_k - m)   (exact 64-bit sum)
  inv_rms = RN(sqrt?(RN(K 2^48 / RN(S)))) * 2^-m          (fp32, IEEE)
(mx_device.cuh, pm_inv_rms; mx_row.cuh, finish_row).  This file restates
those steps with exact rationals and fp32 rounding from its definition and
checks, against the exact value ((1/K) sum_k 2^(p e_k))^(-1/p), the bound
the parity tests rely on: relative error below 2^-22 (K 2^-48 from the
dropped terms, plus three fp32 roundings), for K up to 2^15 blocks (rows of
2^20 elements) and exponent spreads that drop terms.  The GPU parity tests
compare the kernels with the oracle at 1e-6 (about 2^-19.9); the oracle is
within 2^-24 of the exact value (fp64, one fp32 rounding), so kernel and
oracle differ by less than 2^-22 + 2^-24, about a third of the tolerance.
"""
import math
import random
from fractions import Fraction

import pytest

from oracle import bruteforce as bf

F48 = 48


def kernel_model(exps, p):
    """The kernel's steps on the integer exponents of the block scales."""
    K = len(exps)
    m = max(exps)
    S = 0
    for e in exps:
        t = F48 + p * (e - m)
        if t >= 0:
            S += 1 << t
    assert S < 1 << 64
    s = bf.round_to_fp32(Fraction(S))
    q = bf.round_to_fp32(Fraction(K << F48) / s)
    if p == 2:
        q = _sqrt_rn32(q)
    return q * Fraction(2) ** (-m)  # exact: the result stays normal for m <= 125


def _sqrt_rn32(q):
    """Correctly rounded fp32 square root of a positive fp32 rational q,
    decided exactly (compare squares against the rounding boundaries)."""
    approx = bf.round_to_fp32(Fraction(math.sqrt(float(q))))
    # nudge to the fp32 value whose rounding interval holds sqrt(q)
    for _ in range(4):
        e = math.floor(math.log2(approx))
        ulp = Fraction(2) ** (e - 23)
        lo, hi = approx - ulp / 2, approx + ulp / 2
        if lo * lo > q:
            approx -= ulp
        elif hi * hi < q:
            approx += ulp
        else:
            break
    return approx


def rel_err(exps, p):
    """|got / exact - 1| for exact = ((1/K) sum 2^(p e_k))^(-1/p), in exact
    arithmetic: x = got / exact is r mean (p = 1) or r sqrt(mean) (p = 2)
    with r = got 2^m; for p = 2, with d = |x^2 - 1|, |x - 1| = d / (1 + x)
    <= d / (2 - d) since x >= 1 - d."""
    got = kernel_model(exps, p)
    K = len(exps)
    m = max(exps)
    mean = sum(Fraction(2) ** (p * (e - m)) for e in exps) / K
    r = got * Fraction(2) ** m
    if p == 1:
        return abs(r * mean - 1)
    d = abs(r * r * mean - 1)
    return d / (2 - d)


CASES = [
    ("all equal, K = 2^15", [3] * (1 << 15)),
    ("one large block, the rest 24 below", [0] + [-24] * ((1 << 15) - 1)),
    ("one large block, the rest 25 below (dropped for p = 2)", [0] + [-25] * ((1 << 15) - 1)),
    ("one large block, the rest 48 below", [0] + [-48] * ((1 << 15) - 1)),
    ("one large block, the rest 49 below (dropped for p = 1)", [0] + [-49] * ((1 << 15) - 1)),
    ("single block", [-7]),
    ("two blocks far apart", [100, -127]),
    ("E8M0 extremes", [-127, 119]),
]


@pytest.mark.parametrize("name,exps", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("p", [1, 2])
def test_kernel_estimator_within_bound_at_extremes(name, exps, p):
    assert rel_err(exps, p) < Fraction(1, 1 << 22)


@pytest.mark.parametrize("p", [1, 2])
def test_kernel_estimator_within_bound_random(p):
    rng = random.Random(7 + p)
    worst = Fraction(0)
    for _ in range(300):
        K = rng.choice([1, 2, 8, 24, 128, 1000, 4096, 1 << 15])
        spread = rng.choice([0, 3, 12, 24, 30, 60])
        top = rng.randint(-100, 110)
        exps = [top - rng.randint(0, spread) for _ in range(K)]
        worst = max(worst, rel_err(exps, p))
    assert worst < Fraction(1, 1 << 22), float(worst)


def test_tolerance_margin():
    """The parity tests' 1e-6 covers the kernel's bound plus the oracle's own
    rounding with room to spare."""
    assert 2.0 ** -22 + 2.0 ** -24 < 1e-6 / 3

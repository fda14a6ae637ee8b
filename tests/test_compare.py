"""The parity checker itself (oracle.compare), on the CPU: its rounding to
the output types against independent definitions, and each clause of the
two-part check on constructed cases."""
import math
from fractions import Fraction

import numpy as np

from oracle import compare


def exact_round(x: float, bits: int, emin: int) -> float:
    """Round to nearest even with `bits` significant bits, in exact rational
    arithmetic."""
    if x == 0.0:
        return 0.0
    e = max(math.frexp(x)[1] - 1, emin)
    q = Fraction(2) ** (e - bits + 1)
    n = Fraction(x) / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return float(fl * q)


def sample(n=20000, seed=0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal(n) * np.exp2(rng.integers(-30, 8, n).astype(np.float64))


def test_round_to_f16_matches_numpy():
    x = sample()
    x = x[np.abs(x) < 65504]
    assert np.array_equal(compare.round_to_dtype(x, "f16"),
                          x.astype(np.float16).astype(np.float64))


def test_round_to_bf16_and_f32_match_exact_rounding():
    x = sample(4000, 1)
    # halfway cases: a bfloat16 value plus half its spacing, both parities
    b = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -0.75 - 2.0 ** -10, 3.0 * 2.0 ** -130])
    for v in np.concatenate([x, b]):
        assert compare.round_to_dtype(v, "bf16") == exact_round(float(v), 8, -126)
        assert compare.round_to_dtype(v, "f32") == exact_round(float(v), 24, -126)
    assert compare.round_to_dtype(1.0 + 2.0 ** -8, "bf16") == 1.0               # tie to even
    assert compare.round_to_dtype(1.0 + 3 * 2.0 ** -8, "bf16") == 1.0 + 2.0 ** -6
    assert np.array_equal(compare.round_to_dtype(sample(2000, 2), "f32"),
                          sample(2000, 2).astype(np.float32).astype(np.float64))


def test_ulp():
    assert compare.ulp(0.75, "bf16") == 2.0 ** -8
    assert compare.ulp(1.0, "bf16") == 2.0 ** -7
    assert compare.ulp(0.75, "f16") == 2.0 ** -11
    assert compare.ulp(1e-9, "f16") == 2.0 ** -24                             # subnormal spacing


def test_two_part_check_clauses():
    tol = 2e-3
    want = np.array([0.1, 0.7, 0.7, 0.1, 0.3])
    r7 = float(compare.round_to_dtype(0.7, "bf16"))
    got = np.array([0.1 + 0.999 * tol,          # within the bound: passes
                    r7 + 2.0 ** -8,             # above tol, one ulp from the rounded oracle
                    0.7,                        # exact
                    0.1, 0.3])
    p = compare.check(got, want, tol, "bf16")
    assert p.ok and p.n_rounding == 1 and p.max_rounding_ulps == 1.0
    got[1] = r7 + 2 * 2.0 ** -8                  # two ulps away: fails
    p = compare.check(got, want, tol, "bf16")
    assert not p.ok and p.n_bad == 1 and p.worst == (1,)
    got[1] = 0.7
    got[3] = 0.1 + 2.5e-3                        # above tol at a small |out|: one bf16 ulp at
    p = compare.check(got, want, tol, "bf16")   # 0.1 is 2^-11, so not a rounding miss
    assert not p.ok and p.worst == (3,)
    got[3] = float("nan")
    assert not compare.check(got, want, tol, "bf16").ok

"""Parity check of a GPU result against the oracle.

TEST INFRASTRUCTURE, like the rest of this package: the tests and the smoke
check call it; the product path never does.

The decode bound is a max-abs error: 2e-3 for 16-bit caches and 3e-2 for E4M3
caches on unit-variance inputs. The output has the query's type (binary32,
binary16 or bfloat16), rounded to nearest even from the kernel's float32
result, so an output whose magnitude is large enough can miss the bound by its
own rounding alone (a bfloat16 output in [0.5, 1) has a half-unit of 2^-9,
about 1.95e-3). The check therefore has two parts:

1. every element with |gpu - oracle| <= tol passes;
2. an element above tol passes only when it fails through the output
   rounding alone: the GPU value lies within one unit in the last place of the
   output type of round_to_dtype(oracle), the oracle's value rounded to the
   output type.

Elements taking the second part are counted and reported, never silently
absorbed; any other element above tol fails the check.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# significand bits (with the implicit one) and the smallest normal exponent
_FORMATS = {"f32": (24, -126), "f16": (11, -14), "bf16": (8, -126)}


def _binade_exponent(x: np.ndarray, emin: int) -> np.ndarray:
    """floor(log2 |x|), clamped below at the format's smallest normal exponent
    (subnormals share its spacing); frexp is exact, log2 is not."""
    _, e = np.frexp(x)
    return np.maximum(e.astype(np.int64) - 1, emin)


def round_to_dtype(x, dtype: str) -> np.ndarray:
    """x (float64) rounded to nearest even in the output type `dtype`,
    returned as float64. Exact: the scaling by powers of two is exact and
    np.rint rounds half to even."""
    p, emin = _FORMATS[dtype]
    x = np.asarray(x, dtype=np.float64)
    q = np.ldexp(1.0, _binade_exponent(x, emin) - (p - 1))
    return np.rint(x / q) * q


def ulp(x, dtype: str) -> np.ndarray:
    """The spacing of the output type's values in the binade of |x|."""
    p, emin = _FORMATS[dtype]
    x = np.asarray(x, dtype=np.float64)
    return np.ldexp(1.0, _binade_exponent(x, emin) - (p - 1))


@dataclass
class Parity:
    n: int                    # elements compared
    max_err: float            # max |gpu - oracle|
    tol: float
    n_rounding: int           # elements above tol passed by the rounding clause
    max_rounding_ulps: float  # their max |gpu - round(oracle)| in ulps (0 if none)
    n_bad: int                # elements failing both parts
    worst: tuple | None       # index of the worst failing element
    max_abs_out: float
    at_max_out: float = 0.0   # |oracle| at the element of largest error
    at_max_ulps: float = 0.0  # that element's |gpu - round(oracle)| in ulps

    @property
    def ok(self) -> bool:
        return self.n_bad == 0

    def summary(self) -> str:
        s = (f"max err {self.max_err:.3e} (tol {self.tol:g}; at |out| {self.at_max_out:.3f}, "
             f"{self.at_max_ulps:.2f} ulp from the rounded oracle) over {self.n} elements, "
             f"max |out| {self.max_abs_out:.3f}, rounding exceptions {self.n_rounding}")
        if self.n_rounding:
            s += f" (within {self.max_rounding_ulps:.2f} ulp of the rounded oracle)"
        return s


def check(got, want, tol: float, out_dtype: str) -> Parity:
    """Two-part parity check (module docstring). `got` and `want` are float64
    arrays of the same shape; non-finite GPU values always fail."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    err = np.abs(got - want)
    err = np.where(np.isfinite(got), err, np.inf)
    over = err > tol
    n_round, max_ulps, n_bad, worst = 0, 0.0, 0, None
    if over.any():
        r = round_to_dtype(want[over], out_dtype)
        d_ulps = np.abs(got[over] - r) / ulp(r, out_dtype)
        by_rounding = d_ulps <= 1.0
        n_round = int(by_rounding.sum())
        max_ulps = float(d_ulps[by_rounding].max()) if n_round else 0.0
        n_bad = int((~by_rounding).sum())
        if n_bad:
            idx = np.argwhere(over)[~by_rounding]
            bad_err = err[over][~by_rounding]
            worst = tuple(int(i) for i in idx[int(np.argmax(bad_err))])
    at_out = at_ulps = 0.0
    if got.size:
        i = int(np.argmax(err))
        w, g = float(want.flat[i]), float(got.flat[i])
        rw = float(round_to_dtype(w, out_dtype))
        at_out, at_ulps = abs(w), abs(g - rw) / float(ulp(rw, out_dtype))
    return Parity(n=int(got.size), max_err=float(err.max()) if got.size else 0.0, tol=tol,
                  n_rounding=n_round, max_rounding_ulps=max_ulps, n_bad=n_bad, worst=worst,
                  max_abs_out=float(np.abs(want).max()) if want.size else 0.0,
                  at_max_out=at_out, at_max_ulps=at_ulps)

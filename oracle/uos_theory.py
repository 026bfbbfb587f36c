"""Exact rational evaluation of the UOS objective terms -- TEST INFRASTRUCTURE ONLY.

Restates, with Python ``fractions``, the quantities of section 4.1 and
appendices B-C of "MXAttention: Data-Free Optimal Scaling and Pre-Normalization
Quantization for MXFP4 Attention":

* E(x) = integral_0^x (v - Pi(v))^2 dv, the cumulative projection error of the
  nonnegative finite E2M1 grid with saturation at 6 (Eq. 21), integrated piece
  by piece with Eq. 69;
* Delta(q) = E(q) - 8 E(q/2) (Eq. 35), whose sign gives the direction of the
  objective J(q) (Eqs. 36, 80);
* the sign change of Delta on (1/4, inf), located by exact bisection.

The oracle's UOS boundary 7.25 is pinned against :func:`q_star`.
"""
from __future__ import annotations

from fractions import Fraction as F

# Nonnegative finite E2M1 grid (Eq. 20) and its round-to-nearest decision
# thresholds (midpoints of neighbouring grid points, Eq. 68).
GRID = [F(0), F(1, 2), F(1), F(3, 2), F(2), F(3), F(4), F(6)]
THRESHOLDS = [(GRID[i] + GRID[i + 1]) / 2 for i in range(len(GRID) - 1)]


def _pieces():
    """Intervals [a, b) of the magnitude axis and the grid value each maps to."""
    lo = F(0)
    for g, t in zip(GRID[:-1], THRESHOLDS):
        yield lo, t, g
        lo = t
    yield lo, None, GRID[-1]  # saturation: everything above 5 maps to 6


def E(x) -> F:
    """Cumulative projection error E(x), exact for rational x >= 0."""
    x = F(x)
    total = F(0)
    for a, b, r in _pieces():
        if x <= a:
            break
        hi = x if (b is None or x < b) else b
        total += ((hi - r) ** 3 - (a - r) ** 3) / 3  # Eq. 69
    return total


def D(x) -> F:
    """Normalised error D(x) = E(x) / x^3 (Eq. 21)."""
    x = F(x)
    return E(x) / x**3


def delta(q) -> F:
    """Delta(q) = E(q) - 8 E(q/2) (Eq. 35)."""
    q = F(q)
    return E(q) - 8 * E(q / 2)


def q_star(lo=F(6), hi=F(8), iters=80) -> F:
    """Sign change of Delta inside [lo, hi] by exact bisection, snapped to the
    nearest fraction with denominator <= 64."""
    lo, hi = F(lo), F(hi)
    assert delta(lo) < 0 < delta(hi)
    for _ in range(iters):
        mid = (lo + hi) / 2
        if delta(mid) < 0:
            lo = mid
        else:
            hi = mid
    return ((lo + hi) / 2).limit_denominator(64)


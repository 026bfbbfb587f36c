"""Pins of the UOS boundary against the exact derivation printed in "MXAttention".

* E(6) = 7/8, E(3) = 1/8, E(4) = 5/24: Appendix B, Eqs. (70)-(72)
* Delta(q) = -1/8 on [6, 7] and (4q-29)(4q-27)/8 on [7, 8]: Eq. (37) / (73)
* q* = 29/4 is the only sign change: Eq. (38), Eq. (81)
* the last-row quadratic of the sign table has discriminant -18240: Appendix C
* the oracle's UOS boundary equals q*: Theorem 1
Values are read from tests/golden/uos_closed_forms.txt.
"""
import os
from fractions import Fraction as F

import numpy as np

from oracle import uos_theory as T

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "uos_closed_forms.txt")


def _golden():
    out = {}
    with open(GOLDEN) as f:
        for l in f:
            if l.strip() and not l.startswith("#"):
                p = l.split()
                out.setdefault(p[0], []).append(p[1:])
    return out


def test_printed_E_values():
    for x, val in _golden()["E"]:
        assert T.E(F(x)) == F(val)


def test_delta_branches_eq37():
    for q in [F(6), F(25, 4), F(13, 2), F(27, 4), F(7)]:
        assert T.delta(q) == F(-1, 8)
    for q in [F(7), F(29, 4), F(15, 2), F(31, 4), F(8), F(71, 10)]:
        assert T.delta(q) == (4 * q - 29) * (4 * q - 27) / 8


def test_qstar_and_sign_pattern():
    qs = F(_golden()["qstar"][0][0])
    assert T.q_star() == qs == F(29, 4)
    assert T.delta(qs) == 0
    for q in [F(1, 8), F(1, 5), F(1, 4)]:
        assert T.delta(q) == 0
    grid = [F(k, 16) for k in range(5, 116)] + [F(k, 4) for k in range(30, 200)]
    for q in grid:
        d = T.delta(q)
        if q < qs:
            assert d < 0, q
        elif q > qs:
            assert d > 0, q


def test_last_row_discriminant():
    # For q >= 12 both q and q/2 saturate to 6, and 8*Delta is a quadratic in q.
    pts = [F(12), F(14), F(17)]
    ys = [8 * T.delta(q) for q in pts]
    A = np.array([[float(q * q), float(q), 1.0] for q in pts])
    a, b, c = [F(x).limit_denominator(1000) for x in np.linalg.solve(A, np.array([float(y) for y in ys]))]
    for q in [F(20), F(33, 2), F(100)]:
        assert a * q * q + b * q + c == 8 * T.delta(q)
    disc = int(_golden()["discriminant"][0][0])
    assert b * b - 4 * a * c == disc
    assert a > 0  # positive leading coefficient: the branch is strictly positive


def test_oracle_boundary_is_qstar(orc):
    assert orc.uos_qmax() == float(T.q_star())


def test_theory_projection_matches_oracle(orc):
    """The piecewise map used for E(x) agrees with the oracle's projection off the ties."""
    for v in np.linspace(0.01, 9.0, 900):
        if any(abs(v - float(t)) < 1e-9 for t in T.THRESHOLDS):
            continue
        pieces = list(T._pieces())
        r = [p[2] for p in pieces if p[0] <= v and (p[1] is None or v < p[1])][0]
        assert orc.e2m1_value(int(orc.e2m1_code(v))) == float(r)

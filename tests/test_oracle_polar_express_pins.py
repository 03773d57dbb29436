"""Pins of the Polar Express coefficient oracle (``oracle/polar_express.py``).

The pages (DMuon "API Reference", section *POLAR_EXPRESS_COEFFICIENTS*) fix
the method and the safety factor but print no values, so the table is pinned
by what the method's definition and the mathematics fix, each checked by
brute force rather than by rerunning the Remez routine:

* each step's polynomial is the best uniform approximation of 1 on its
  interval: by the alternation theorem for the Haar system {x, x^3, x^5} on
  (0, inf), that holds iff 1 - p reaches its maximum modulus with alternating
  signs at four points -- checked on a dense grid;
* no nearby polynomial does better (random perturbations, dense grid);
* the steps chain: each interval is the image of the previous one, and the
  composed polynomial maps [1e-3, 1] into [1 - E_last, 1 + E_last];
* a closed-form limit: as the interval shrinks to the point 1 the best
  quintic tends to the one with p(1) = 1, p'(1) = p''(1) = 0, which is
  (15 x - 10 x^3 + 3 x^5) / 8;
* the safety factor is the printed formula ``(a/s, b/s^3, c/s^5)``, i.e. p(x/s).

Planted mistakes (no interval update, a two-point fit, the wrong safety
powers) are applied to copies here and must fail.
"""
import numpy as np
import pytest

from oracle import polar_express as pe

GRID = 200001


def _grid(lo, hi):
    return np.linspace(lo, hi, GRID)


def _max_err(row, lo, hi):
    return float(np.max(np.abs(1.0 - pe.quintic(_grid(lo, hi), *row))))


def _alternation_points(row, lo, hi):
    """Local extrema of 1 - p on a dense grid, endpoints included."""
    x = _grid(lo, hi)
    r = 1.0 - pe.quintic(x, *row)
    idx = [0]
    for i in range(1, len(x) - 1):
        if (r[i] - r[i - 1]) * (r[i + 1] - r[i]) < 0:
            idx.append(i)
    idx.append(len(x) - 1)
    return x[idx], r[idx]


@pytest.mark.parametrize("interval", [(1e-3, 1.0), (0.05, 1.9), (0.3, 1.0), (0.5, 1.5), (0.9, 1.1)])
def test_minimax_equioscillates(interval):
    lo, hi = interval
    a, b, c, E = pe.minimax_quintic(lo, hi)
    xs, rs = _alternation_points((a, b, c), lo, hi)
    assert len(xs) == 4
    assert np.all(np.abs(np.abs(rs) - E) <= 1e-9 * max(E, 1e-300) + 1e-14)
    assert np.all(np.sign(rs) == np.array([1, -1, 1, -1]))
    assert abs(_max_err((a, b, c), lo, hi) - E) <= 1e-9 * E + 1e-14


@pytest.mark.parametrize("interval", [(1e-3, 1.0), (0.2, 1.8)])
def test_no_nearby_polynomial_does_better(interval):
    lo, hi = interval
    a, b, c, E = pe.minimax_quintic(lo, hi)
    rng = np.random.default_rng(11)
    base = _max_err((a, b, c), lo, hi)
    for _ in range(200):
        d = rng.standard_normal(3) * 1e-4 * np.array([abs(a), abs(b), abs(c)])
        assert _max_err((a + d[0], b + d[1], c + d[2]), lo, hi) >= base * (1 - 1e-9)


def test_steps_chain_and_compose():
    steps = pe.polar_express_steps(5)
    lo, hi = pe.LOWER0, pe.UPPER0
    Es = []
    for row, (l, u), E in steps:
        assert (l, u) == pytest.approx((lo, hi), rel=0, abs=1e-15)
        assert pe.quintic(l, *row) == pytest.approx(1 - E, abs=1e-12)
        assert float(np.max(pe.quintic(_grid(l, u), *row))) == pytest.approx(1 + E, abs=1e-9)
        lo, hi = 1 - E, 1 + E
        Es.append(E)
    assert all(e1 < e0 for e0, e1 in zip(Es, Es[1:]))      # each step tightens
    x = np.geomspace(pe.LOWER0, 1.0, 20001)
    y = x.copy()
    for row, _, _ in steps:
        y = pe.quintic(y, *row)
    assert np.all(np.abs(1 - y) <= Es[-1] * (1 + 1e-9))


def test_narrow_interval_tends_to_the_osculating_quintic():
    a, b, c, E = pe.minimax_quintic(0.999, 1.0)
    assert E < 1e-9
    assert (a, b, c) == pytest.approx((15 / 8, -10 / 8, 3 / 8), abs=2e-3)
    # and that limit polynomial really is flat to second order at 1
    p = lambda x: (15 * x - 10 * x ** 3 + 3 * x ** 5) / 8  # noqa: E731
    h = 1e-4
    assert p(1.0) == pytest.approx(1.0, abs=1e-15)
    assert (p(1 + h) - p(1 - h)) / (2 * h) == pytest.approx(0.0, abs=1e-7)
    assert (p(1 + h) - 2 * p(1.0) + p(1 - h)) / h ** 2 == pytest.approx(0.0, abs=1e-4)


def test_longer_tables_extend_shorter_ones():
    """Each row depends only on the rows before it, so a longer table starts
    with the shorter one; past the point where the interval is within 1e-7 of
    1 the rows are the limit quintic (15/8, -10/8, 3/8)."""
    short, long_ = pe.polar_express_steps(5), pe.polar_express_steps(10)
    for (r1, i1, e1), (r2, i2, e2) in zip(short, long_):
        assert r1 == r2 and i1 == i2 and e1 == e2
    tail = [r for r, (l, u), _ in long_ if l >= 1 - pe.TINY and u <= 1 + pe.TINY]
    assert tail and all(r == (15 / 8, -10 / 8, 3 / 8) for r in tail)
    assert long_[-1][2] < 1e-15


def test_safety_factor_is_p_of_x_over_s():
    rows = pe.polar_express_rows(5)
    raw = [r for r, _, _ in pe.polar_express_steps(5)]
    x = np.linspace(0.0, 2.0, 101)
    for r, q in zip(rows, raw):
        assert np.allclose(pe.quintic(x, *r), pe.quintic(x / 1.05, *q), rtol=0, atol=1e-12)
    assert pe.SAFETY_FACTOR == 1.05


def test_table_drives_the_newton_schulz_oracle():
    """The derived table run through the direct oracle orthogonalises a
    matrix whose normalised singular values span [2e-3, 0.66] (inside the
    design interval [1e-3, 1] after the safety factor's 1/1.05)."""
    import oracle
    rng = np.random.default_rng(12)
    U, _ = np.linalg.qr(rng.standard_normal((40, 40)))
    V, _ = np.linalg.qr(rng.standard_normal((60, 40)))
    s = np.geomspace(1.0, 3e-3, 40) * 0.1
    G = (U * s) @ V.T
    sig = s / np.linalg.norm(s)
    assert sig.min() / 1.05 > pe.LOWER0 and sig.max() <= 1.0
    O = oracle.newton_schulz(G, 5, coeffs=pe.polar_express_rows(5))
    sv = np.linalg.svd(O, compute_uv=False)
    assert sv.min() > 0.8 and sv.max() < 1.15, (sv.min(), sv.max())


# ------------------------------------------------------------ planted slips

def test_planted_slips_fail_the_pins():
    # (1) keeping the starting interval instead of following the image
    rows_stuck = [pe.minimax_quintic(pe.LOWER0, pe.UPPER0)[:3]] * 2
    x = np.geomspace(pe.LOWER0, 1.0, 2001)
    y = pe.quintic(pe.quintic(x, *rows_stuck[0]), *rows_stuck[1])
    E2 = pe.polar_express_steps(2)[-1][2]
    assert np.max(np.abs(1 - y)) > 1.5 * E2
    # (2) a fit that only matches the endpoints does not equioscillate
    lo, hi = 0.1, 1.0
    M = np.array([[lo, lo ** 3, lo ** 5], [hi, hi ** 3, hi ** 5], [0.5, 0.125, 0.03125]])
    row = np.linalg.solve(M, np.ones(3))
    xs, rs = _alternation_points(row, lo, hi)
    assert not (len(xs) == 4 and np.allclose(np.abs(rs), np.abs(rs[0]), rtol=1e-6))
    # (3) the safety factor applied with the wrong powers is not p(x/s)
    (a, b, c), _, _ = pe.polar_express_steps(1)[0]
    wrong = (a / 1.05, b / 1.05 ** 2, c / 1.05 ** 3)
    assert not np.allclose(pe.quintic(0.7, *wrong), pe.quintic(0.7 / 1.05, a, b, c), atol=1e-6)

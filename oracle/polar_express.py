"""fp64 oracle of Polar Express coefficient tables (test infrastructure).

Test infrastructure only, like the rest of ``oracle/``: the test-suite, the
smoke check and the CPU leg of ``bench.py`` may use it; the CUDA library
never does, and this module imports nothing from it.

What the pages fix (DMuon "API Reference", section
*POLAR_EXPRESS_COEFFICIENTS*): the Gram backend's default five-step table
comes from Polar Express (arXiv:2505.16932) and is the unmodified table with
a safety factor s = 1.05 applied as ``(a / s, b / s**3, c / s**5)`` per row,
i.e. ``p(x / s)``.  The unmodified values are not printed.

The method (the paper's construction, restated): with every singular value
of the normalised input known to lie in ``[l, u]``, each step takes the odd
quintic ``p(x) = a x + b x**3 + c x**5`` that minimises
``max over x in [l, u] of |1 - p(x)|`` (a Chebyshev approximation of the
constant 1 by ``{x, x**3, x**5}``), and the next step's interval is the image
``[1 - E, 1 + E]``, E being that minimal maximum error.  The best
approximation equioscillates: ``1 - p`` takes the values ``+E, -E, +E, -E``
at four points ``l = x0 < x1 < x2 < x3 = u`` and nowhere exceeds ``|E|``.

Readings of points the pages leave open ("parity unpinned": the pages print
no values to compare with):

* the starting interval is ``[1e-3, 1]`` (u = 1 because the Frobenius-
  normalised input has spectral norm at most 1; l = 1e-3 as the smallest
  singular value the table is meant to lift);
* no other modification than the printed safety factor is applied;
* once the interval has shrunk to within ``TINY`` of the point 1 (half-width
  at most 1e-7, reached after about six steps from ``[1e-3, 1]``) the exchange
  has nothing left to resolve in fp64; such steps take the construction's
  limit, the quintic with ``p(1) = 1, p'(1) = p''(1) = 0``, i.e.
  ``(15/8, -10/8, 3/8)``, which differs from the minimax row by about the
  half-width.

The minimax step is computed by the Remez exchange: solve for ``a, b, c, E``
on a four-point reference, move the reference to the local extrema of
``1 - p`` (the two interior ones are the positive roots of
``p'(x) = a + 3 b x**2 + 5 c x**4``, a quadratic in ``x**2``), repeat.  The
pins in ``tests/test_oracle_polar_express_pins.py`` check the result by the
alternation property on a dense grid, not by rerunning this routine.
"""

import numpy as np

# DMuon "API Reference", section POLAR_EXPRESS_COEFFICIENTS: safety factor.
SAFETY_FACTOR = 1.05
# Starting interval of the singular values (readings above).
LOWER0, UPPER0 = 1e-3, 1.0
# Half-width below which a step takes the limit row (readings above).
TINY = 1e-7
LIMIT_ROW = (15.0 / 8.0, -10.0 / 8.0, 3.0 / 8.0)


def quintic(x, a, b, c):
    """``p(x) = a x + b x**3 + c x**5``."""
    x = np.asarray(x, np.float64)
    x2 = x * x
    return x * (a + x2 * (b + c * x2))


def interior_extrema(a, b, c, lo, hi):
    """Points of ``(lo, hi)`` where ``p'(x) = a + 3 b x**2 + 5 c x**4`` vanishes."""
    ys = np.roots([5.0 * c, 3.0 * b, a]) if c != 0.0 else (np.roots([3.0 * b, a]) if b != 0.0 else [])
    xs = []
    for y in np.atleast_1d(ys):
        if abs(np.imag(y)) > 1e-12 * max(1.0, abs(y)):
            continue
        y = float(np.real(y))
        if y > 0.0:
            x = np.sqrt(y)
            if lo < x < hi:
                xs.append(x)
    return sorted(xs)


def minimax_quintic(lo, hi, max_iter=200):
    """``(a, b, c, E)``: the odd quintic with the least ``max |1 - p|`` on
    ``[lo, hi]`` and that error (``E > 0``; ``1 - p(lo) = +E``)."""
    if not 0.0 < lo < hi:
        raise ValueError("need 0 < lo < hi")
    signs = np.array([1.0, -1.0, 1.0, -1.0])
    k = np.arange(4)
    ref = 0.5 * (lo + hi) - 0.5 * (hi - lo) * np.cos(np.pi * k / 3.0)
    prev = None
    for _ in range(max_iter):
        M = np.stack([ref, ref ** 3, ref ** 5, signs], axis=1)
        a, b, c, E = np.linalg.solve(M, np.ones(4))
        inner = interior_extrema(a, b, c, lo, hi)
        if len(inner) != 2:
            raise RuntimeError("Remez reference lost its two interior extrema on [%g, %g]" % (lo, hi))
        ref = np.array([lo, inner[0], inner[1], hi])
        err = np.max(np.abs(1.0 - quintic(ref, a, b, c)))
        if prev is not None and abs(err - abs(E)) <= 1e-15 * max(1.0, err) and abs(E - prev) <= 1e-16:
            break
        prev = E
    if E <= 0.0:
        raise RuntimeError("unexpected alternation sign on [%g, %g]" % (lo, hi))
    return float(a), float(b), float(c), float(E)


def polar_express_steps(steps=5, lo=LOWER0, hi=UPPER0):
    """Unmodified rows and the interval each step was built for:
    ``[((a, b, c), (l, u), E), ...]``; the next interval is ``[1 - E, 1 + E]``."""
    out = []
    for _ in range(steps):
        if lo >= 1.0 - TINY and hi <= 1.0 + TINY:
            row = LIMIT_ROW
            E = float(max(abs(1.0 - quintic(lo, *row)), abs(1.0 - quintic(hi, *row))))
        else:
            a, b, c, E = minimax_quintic(lo, hi)
            row = (a, b, c)
        out.append((row, (lo, hi), E))
        lo, hi = 1.0 - E, 1.0 + E
    return out


def polar_express_rows(steps=5, lo=LOWER0, hi=UPPER0, safety=SAFETY_FACTOR):
    """The coefficient table: unmodified rows with the safety factor applied
    as ``(a / s, b / s**3, c / s**5)``."""
    s = float(safety)
    return [(a / s, b / s ** 3, c / s ** 5) for (a, b, c), _, _ in polar_express_steps(steps, lo, hi)]

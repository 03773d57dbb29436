"""fp64 oracle of Gram-space Newton-Schulz with restarts (test infrastructure).

Test infrastructure only, like the rest of ``oracle/``: the test-suite, the
smoke check and the CPU leg of ``bench.py`` may use it; the CUDA library
never does, and this module imports nothing from it.

What the pages fix (DMuon "API Reference", sections *NewtonSchulz*,
*newton_schulz*, *gram_newton_schulz*, *gram_newton_schulz_factors*):

* the Gram backend iterates on the Gram matrix instead of the full
  matrix, with per-step coefficients and restarts;
* the result is the normalised, possibly transposed input left-multiplied
  by one Gram factor per restart window (``gram_newton_schulz_factors``
  returns those factors, the transposed flag and the normaliser
  ``norm + eps`` under the orientation rule of the direct backend);
* ``restart_iterations`` lists restart positions, default ``[2]``.

The algebra the pages leave to the reader, written out here: one quintic
step ``X' = a X + b (X X^T) X + c (X X^T)^2 X`` is ``X' = Z X`` with
``Z = a I + b R + c R^2`` and ``R = X X^T``.  ``Z`` is a polynomial in
``R``, so it is symmetric and commutes with ``R``; hence after the step
``R' = X' X'^T = Z R Z`` and, over a window of steps started from ``X_s``,
``X = Q X_s`` with ``Q = Z_last ... Z_first``.  A window therefore needs
only m x m products; at a restart the iterate is formed explicitly
(``X = Q X``), its Gram matrix is recomputed and ``Q`` starts again from
the identity.

Readings of points the pages leave open:

* a restart position ``k`` means "before step ``k`` (0-based)"; positions
  ``<= 0`` or ``>= ns_steps`` start no new window;
* the coefficients default to the Polar Express table, as the pages state for
  ``gram_newton_schulz`` ("Defaults to POLAR_EXPRESS_COEFFICIENTS"); its
  values are not printed, so the default is the table ``oracle.polar_express``
  derives by the method's construction (``ns_steps`` rows; its own readings and
  pins live there).

In exact arithmetic the Gram backend equals the direct one for every
restart set; the pins in ``tests/test_oracle_gram_pins.py`` check that,
the SVD closed form, and the structure of the factors.
"""

import numpy as np

from .polar_express import polar_express_rows
from .step import DEFAULT_EPS, coefficient_rows, frobenius_normalize, momentum_update, \
    nesterov_input, orient, update_scale, apply_update


def gram_rows(ns_steps, coeffs=None):
    """Per-step rows of the Gram backend: ``coeffs`` if given, else the
    Polar Express table of ``ns_steps`` rows (DMuon "API Reference", section
    *gram_newton_schulz*: coefficients default to POLAR_EXPRESS_COEFFICIENTS)."""
    if coeffs is None and ns_steps > 0:
        coeffs = polar_express_rows(ns_steps)
    return coefficient_rows(ns_steps, coeffs)


def restart_windows(ns_steps, restarts=(2,)):
    """Step ranges ``[(start, end), ...]`` of the restart windows.

    Positions outside ``(0, ns_steps)`` are ignored (reading above);
    duplicates collapse.  ``ns_steps == 0`` gives no window.
    """
    cuts = sorted({int(k) for k in (restarts or ()) if 0 < int(k) < ns_steps})
    bounds = [0] + cuts + [ns_steps]
    return [(bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1) if bounds[i + 1] > bounds[i]]


def gram_window_factor(X, rows):
    """Gram factor of one window: ``Q = Z_last ... Z_first`` for the steps
    ``rows`` started from iterate ``X`` (m x n), using only m x m products:
    ``R = X X^T``; per step ``Z = a I + b R + c R R``, ``Q <- Z Q``,
    ``R <- Z R Z``."""
    X = np.asarray(X, np.float64)
    m = X.shape[0]
    eye = np.eye(m)
    R = X @ X.T
    Q = eye.copy()
    for a, b, c in rows:
        Z = a * eye + b * R + c * (R @ R)
        Q = Z @ Q
        R = Z @ R @ Z
    return Q


def gram_newton_schulz_factors(G, ns_steps=5, coeffs=None, restarts=(2,), eps=DEFAULT_EPS):
    """Factors of the Gram backend: ``(segments, transposed, normaliser)``.

    ``segments`` holds one m x m factor per restart window, in order; the
    output is ``O = Q_last ... Q_1 X0`` with ``X0`` the normalised oriented
    input, transposed back when ``transposed``.
    """
    rows = gram_rows(ns_steps, coeffs)
    Y, transposed = orient(G)
    X, normaliser = frobenius_normalize(Y, eps)
    segments = []
    for start, end in restart_windows(ns_steps, restarts):
        Q = gram_window_factor(X, rows[start:end])
        segments.append(Q)
        X = Q @ X   # the next window starts from the explicit iterate
    return segments, transposed, normaliser


def gram_newton_schulz(G, ns_steps=5, coeffs=None, restarts=(2,), eps=DEFAULT_EPS):
    """Orthogonalised ``O`` (shape of ``G``) by the Gram backend."""
    segments, transposed, normaliser = gram_newton_schulz_factors(G, ns_steps, coeffs, restarts, eps)
    Y, _ = orient(G)
    X = Y / normaliser
    for Q in segments:
        X = Q @ X
    return X.T.copy() if transposed else X


def muon_step_gram(W, G, M, lr=0.02, mu=0.95, wd=0.0, ns_steps=5, coeffs=None, restarts=(2,),
                   nesterov=True, eps=DEFAULT_EPS, scale_mode=0):
    """One owner-side Muon step with the Gram backend: the direct step of
    ``oracle.step.muon_step`` with its Newton-Schulz call replaced."""
    W = np.asarray(W, np.float64)
    rows_, cols_ = W.shape
    M_new = momentum_update(M, G, mu)
    U = nesterov_input(G, M_new, mu, nesterov)
    O = gram_newton_schulz(U, ns_steps, coeffs, restarts, eps)
    scale = update_scale(rows_, cols_, scale_mode)
    return {"W": apply_update(W, O, lr, wd, scale), "M": M_new, "O": O, "scale": scale}

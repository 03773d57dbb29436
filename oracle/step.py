"""fp64 oracle of the owner-side Muon step (test infrastructure only).

Test infrastructure: only tests/, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use this module.  It shares no code, table or
helper with the CUDA library; the coefficient table below is typed here
independently from the pages.

Notation (DMuon "API Reference", sections *Muon* and *direct_newton_schulz*):
``W, G, M`` are one weight matrix, its gradient and its momentum buffer, all
``rows x cols``.  ``mu`` is ``momentum``, ``lr`` the Muon learning rate,
``wd`` the Muon weight decay, ``(a_k, b_k, c_k)`` the per-step quintic
coefficients.

Every array operation is float64.  A dense ``@`` is the only library
primitive; there is no blocking, fusion or reordering beyond the steps as
the pages state them.

Readings of points the pages leave open:

1. Nesterov uses the buffer *after* this step's momentum update
   (``U = G + mu * M_new``); the pre-update reading would make Nesterov the
   same as plain momentum.
2. With no coefficient table given, the printed ``YOU_COEFFICIENTS`` rows
   are used; for more than five steps the last row repeats ("parity
   unpinned": the pages print no longer table).
3. The normaliser is ``||Y||_F + eps`` of the oriented Nesterov input.
4. The matrix is transposed iff rows > cols; square matrices are not.
5. The update scale is not stated on the pages ("parity unpinned");
   ``scale_mode`` 0 = ``sqrt(max(1, rows/cols))``, 1 = ``1``,
   2 = ``0.2 * sqrt(max(rows, cols))``.
6. Weight decay is decoupled and multiplicative:
   ``W' = (1 - lr*wd) * W - lr * scale * O``.
"""

import numpy as np

# DMuon "API Reference", section YOU_COEFFICIENTS: five (a, b, c) rows.
YOU_COEFFICIENTS = (
    (4.0848, -6.8946, 2.927),
    (3.9505, -6.3029, 2.6377),
    (3.7418, -5.5913, 2.3037),
    (2.8769, -3.1427, 1.2046),
    (2.8366, -3.0525, 1.2012),
)

# DMuon "API Reference", section direct_newton_schulz: default eps.
DEFAULT_EPS = 1e-7


def coefficient_rows(ns_steps, coeffs=None):
    """Per-step (a, b, c) rows for ``ns_steps`` iterations.

    DMuon "API Reference", section *direct_newton_schulz*: the length of the
    coefficient list sets the number of iterations.  With ``coeffs=None`` the
    ``YOU_COEFFICIENTS`` table is used and its last row repeats past five
    steps (reading 2, parity unpinned beyond five).
    """
    if ns_steps < 0:
        raise ValueError("ns_steps must be >= 0")
    if coeffs is not None:
        rows = [tuple(float(v) for v in r) for r in coeffs]
        if len(rows) != ns_steps or any(len(r) != 3 for r in rows):
            raise ValueError("coeffs must hold ns_steps rows of (a, b, c)")
        return rows
    table = [tuple(r) for r in YOU_COEFFICIENTS]
    return [table[min(k, len(table) - 1)] for k in range(ns_steps)]


def momentum_update(M, G, mu):
    """Momentum buffer update ``M_new = mu * M + G``.

    DMuon "API Reference", section *Muon*: ``momentum`` is the coefficient of
    the dedicated-parameter momentum buffer.
    """
    return mu * np.asarray(M, np.float64) + np.asarray(G, np.float64)


def nesterov_input(G, M_new, mu, nesterov=True):
    """Input of Newton-Schulz: ``G + mu * M_new`` (Nesterov) or ``M_new``.

    DMuon "API Reference", section *Muon*, argument ``nesterov``: the
    Newton-Schulz input is the gradient plus momentum times the buffer.
    """
    G = np.asarray(G, np.float64)
    M_new = np.asarray(M_new, np.float64)
    return G + mu * M_new if nesterov else M_new.copy()


def orient(U):
    """Orientation rule: work on ``U^T`` iff rows > cols.

    DMuon "API Reference", section *gram_newton_schulz_factors*: the
    normaliser and the iteration use the possibly transposed view.
    Returns ``(Y, transposed)``.
    """
    U = np.asarray(U, np.float64)
    if U.shape[0] > U.shape[1]:
        return U.T.copy(), True
    return U.copy(), False


def frobenius_normalize(Y, eps=DEFAULT_EPS):
    """``X0 = Y / (||Y||_F + eps)``.

    DMuon "API Reference", sections *direct_newton_schulz* (``eps``) and
    *gram_newton_schulz_factors* (normaliser = ``G.norm() + eps``).
    Returns ``(X0, normaliser)``.
    """
    Y = np.asarray(Y, np.float64)
    norm = np.sqrt(np.sum(Y * Y)) + eps
    return Y / norm, norm


def newton_schulz_direct(X, rows):
    """Direct (parameter-space) quintic Newton-Schulz.

    DMuon "API Reference", section *direct_newton_schulz*: for each step k,
    ``X <- a_k X + b_k (X X^T) X + c_k (X X^T)^2 X``, written as
    ``A = X X^T``, ``B = b_k A + c_k A A``, ``X = a_k X + B X``.
    """
    X = np.asarray(X, np.float64)
    for a, b, c in rows:
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X


def newton_schulz(G, ns_steps=5, coeffs=None, eps=DEFAULT_EPS):
    """Orthogonalised matrix ``O`` of the same shape as ``G``.

    Orientation, normalisation, iteration, then orientation back, as in
    DMuon "API Reference", section *direct_newton_schulz*.
    """
    rows = coefficient_rows(ns_steps, coeffs)
    Y, transposed = orient(G)
    X0, _ = frobenius_normalize(Y, eps)
    X = newton_schulz_direct(X0, rows)
    return X.T.copy() if transposed else X


def update_scale(rows, cols, scale_mode=0):
    """Scale applied to the Newton-Schulz output in the weight update.

    The pages call this step only "update" (DMuon "HSDP Training", section
    *What Happens Under the Hood*) and give no factor: parity unpinned.
    Mode 0 is the original Muon factor ``sqrt(max(1, rows/cols))``; mode 1
    is no scaling; mode 2 is the Moonlight factor ``0.2*sqrt(max(rows,cols))``
    (Moonlight is the formulation the *Muon* argument notes name).
    """
    if scale_mode == 0:
        return float(np.sqrt(max(1.0, rows / cols)))
    if scale_mode == 1:
        return 1.0
    if scale_mode == 2:
        return float(0.2 * np.sqrt(max(rows, cols)))
    raise ValueError("scale_mode must be 0, 1 or 2")


def apply_update(W, O, lr, wd, scale):
    """Decoupled weight decay then the scaled step:
    ``W' = (1 - lr*wd) * W - lr * scale * O`` (reading 6)."""
    W = np.asarray(W, np.float64)
    return (1.0 - lr * wd) * W - lr * scale * np.asarray(O, np.float64)


def muon_step(W, G, M, lr=0.02, mu=0.95, wd=0.0, ns_steps=5, coeffs=None,
              nesterov=True, eps=DEFAULT_EPS, scale_mode=0):
    """One owner-side Muon step on one matrix.

    Order of the steps (DMuon "HSDP Training", *What Happens Under the
    Hood*; DMuon "API Reference", *Muon* and *direct_newton_schulz*):
    momentum, Nesterov input, orientation, normalisation, ``ns_steps``
    quintic iterations, orientation back, decoupled decay and scaled update.

    Returns a dict with float64 arrays ``W`` (new weight), ``M`` (new
    momentum buffer), ``O`` (Newton-Schulz output, shape of ``W``) and the
    float ``scale``.
    """
    W = np.asarray(W, np.float64)
    rows_, cols_ = W.shape
    M_new = momentum_update(M, G, mu)
    U = nesterov_input(G, M_new, mu, nesterov)
    O = newton_schulz(U, ns_steps, coeffs, eps)
    scale = update_scale(rows_, cols_, scale_mode)
    W_new = apply_update(W, O, lr, wd, scale)
    return {"W": W_new, "M": M_new, "O": O, "scale": scale}

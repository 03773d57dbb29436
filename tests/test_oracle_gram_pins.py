"""Pins of the Gram-space Newton-Schulz oracle (``oracle/gram.py``).

The Gram backend is an algebraic rewrite of the direct iteration (DMuon
"API Reference", sections *gram_newton_schulz* and
*gram_newton_schulz_factors*), so in fp64 it must reproduce:

* the direct oracle, for every restart set (the direct oracle is itself
  pinned to the SVD closed form in test_oracle_pins.py);
* the SVD closed form ``U p(S) V^T`` directly, with ``p`` the composed
  scalar quintics applied to the normalised singular values;
* the structure the pages describe for the factors: one symmetric m x m
  factor per restart window, each commuting with its window's Gram matrix,
  whose product applied to the normalised oriented input gives the output,
  with the normaliser ``norm + eps``.

Planted mistakes (a one-sided Gram update, a restart that keeps the old Gram
matrix, a restart that keeps the old factor) are applied to a copy of the
window routine here and must fail these pins.
"""
import numpy as np
import pytest

import oracle
from oracle import gram as og
from oracle import polar_express as pe

SHAPES = [(7, 13), (13, 7), (16, 16), (5, 40), (40, 5), (1, 9), (9, 1), (3, 3)]
RESTARTS = [(), (1,), (2,), (3,), (1, 3), (2, 4), (1, 2, 3, 4)]


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def _svd_closed_form(G, rows, eps=1e-7):
    Y = G.T if G.shape[0] > G.shape[1] else G
    U, S, Vt = np.linalg.svd(Y, full_matrices=False)
    s = S / (np.sqrt(np.sum(Y * Y)) + eps)
    for a, b, c in rows:
        s = a * s + b * s ** 3 + c * s ** 5
    O = (U * s) @ Vt
    return O.T if G.shape[0] > G.shape[1] else O


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("restarts", RESTARTS)
def test_gram_equals_direct(shape, restarts):
    G = np.random.default_rng(hash((shape, restarts)) % 2**32).standard_normal(shape)
    # the Gram default (the Polar Express table) and the printed table
    got = og.gram_newton_schulz(G, 5, restarts=restarts)
    ref = oracle.newton_schulz(G, 5, coeffs=pe.polar_express_rows(5))
    assert got.shape == G.shape
    assert _rel(got, ref) <= 1e-10
    got = og.gram_newton_schulz(G, 5, coeffs=oracle.coefficient_rows(5), restarts=restarts)
    assert _rel(got, oracle.newton_schulz(G, 5)) <= 1e-10


def test_gram_default_table_is_polar_express():
    """DMuon "API Reference", section gram_newton_schulz: the coefficients
    default to POLAR_EXPRESS_COEFFICIENTS, here the table derived by
    oracle.polar_express (its own pins), of ns_steps rows."""
    G = np.random.default_rng(9).standard_normal((10, 17))
    for ns in (1, 5, 7):
        assert og.gram_rows(ns) == [tuple(r) for r in pe.polar_express_rows(ns)]
        a = og.gram_newton_schulz(G, ns)
        b = og.gram_newton_schulz(G, ns, coeffs=pe.polar_express_rows(ns))
        assert np.array_equal(a, b)
    assert og.gram_rows(0) == []


@pytest.mark.parametrize("shape", [(6, 11), (11, 6), (8, 8)])
def test_gram_matches_svd_closed_form(shape):
    rng = np.random.default_rng(7)
    G = rng.standard_normal(shape)
    for ns in (1, 3, 5, 7):
        rows = pe.polar_express_rows(ns)
        got = og.gram_newton_schulz(G, ns, restarts=(2,))
        assert _rel(got, _svd_closed_form(G, rows)) <= 1e-10, ns
    coeffs = [(3.0, -3.2, 1.2), (2.5, -2.0, 0.5), (1.875, -1.25, 0.375)]
    got = og.gram_newton_schulz(G, 3, coeffs=coeffs, restarts=(1,))
    assert _rel(got, _svd_closed_form(G, coeffs)) <= 1e-10


def test_restart_windows():
    assert og.restart_windows(5, (2,)) == [(0, 2), (2, 5)]
    assert og.restart_windows(5, ()) == [(0, 5)]
    assert og.restart_windows(5, None) == [(0, 5)]
    assert og.restart_windows(5, (0, 5, 9, -1)) == [(0, 5)]
    assert og.restart_windows(5, (3, 1, 3)) == [(0, 1), (1, 3), (3, 5)]
    assert og.restart_windows(0, (2,)) == []
    assert og.restart_windows(1, (2,)) == [(0, 1)]


def test_restart_positions_outside_the_steps_change_nothing():
    G = np.random.default_rng(3).standard_normal((9, 14))
    base = og.gram_newton_schulz(G, 5, restarts=())
    for r in [(0,), (5,), (9,), (0, 5)]:
        assert np.array_equal(og.gram_newton_schulz(G, 5, restarts=r), base)


def test_zero_steps_is_the_normalised_input():
    G = np.random.default_rng(4).standard_normal((6, 4))
    got = og.gram_newton_schulz(G, 0)
    assert np.allclose(got, G / (np.linalg.norm(G) + 1e-7), rtol=0, atol=1e-15)


@pytest.mark.parametrize("shape", [(7, 13), (13, 7)])
def test_factor_structure(shape):
    G = np.random.default_rng(5).standard_normal(shape)
    segs, transposed, normaliser = og.gram_newton_schulz_factors(G, 5, restarts=(2,))
    assert transposed == (shape[0] > shape[1])
    assert abs(normaliser - (np.linalg.norm(G) + 1e-7)) <= 1e-12 * normaliser
    assert len(segs) == 2
    Y = G.T if transposed else G
    X = Y / normaliser
    for Q in segs:
        m = Y.shape[0]
        assert Q.shape == (m, m)
        assert np.allclose(Q, Q.T, rtol=0, atol=1e-12 * np.abs(Q).max())
        R = X @ X.T
        assert np.linalg.norm(Q @ R - R @ Q) <= 1e-12 * np.linalg.norm(Q) * np.linalg.norm(R)
        X = Q @ X
    O = og.gram_newton_schulz(G, 5, restarts=(2,))
    assert _rel(X.T if transposed else X, O) <= 1e-14


def test_single_window_factor_is_the_composed_polynomial_of_r():
    """Without restarts the factor is q(R0) with q composed from the steps:
    on R0's eigenvectors it multiplies each normalised singular value by
    p(s)/s (p the composed quintic)."""
    G = np.random.default_rng(6).standard_normal((5, 12))
    (Q,), _, nrm = og.gram_newton_schulz_factors(G, 5, restarts=())
    X0 = G / nrm
    U, S, _ = np.linalg.svd(X0, full_matrices=False)
    s = S.copy()
    for a, b, c in pe.polar_express_rows(5):
        s = a * s + b * s ** 3 + c * s ** 5
    assert _rel(Q, (U * (s / S)) @ U.T) <= 1e-10


def test_muon_step_gram_equals_direct_step():
    rng = np.random.default_rng(8)
    for shape in [(12, 20), (20, 12)]:
        W, G, M = (rng.standard_normal(shape) for _ in range(3))
        for kw in [dict(), dict(nesterov=False), dict(wd=0.1, scale_mode=2), dict(ns_steps=3)]:
            rows = oracle.coefficient_rows(kw.get("ns_steps", 5))  # the direct default on both
            a = og.muon_step_gram(W, G, M, lr=0.05, mu=0.9, coeffs=rows, **kw)
            b = oracle.muon_step(W, G, M, lr=0.05, mu=0.9, **kw)
            assert np.array_equal(a["M"], b["M"])
            assert _rel(a["W"] - W, b["W"] - W) <= 1e-10
            assert a["scale"] == b["scale"]


# ------------------------------------------------------------ planted slips

def _one_sided_r(X, rows):
    m = X.shape[0]
    R, Q = X @ X.T, np.eye(m)
    for a, b, c in rows:
        Z = a * np.eye(m) + b * R + c * (R @ R)
        Q = Z @ Q
        R = Z @ R          # slip: R' = Z R instead of Z R Z
    return Q


def _run_with(window, G, restarts=(2,), stale=None):
    rows = oracle.coefficient_rows(5)
    Y, tr = oracle.orient(G)
    X, _ = oracle.frobenius_normalize(Y)
    X0 = X.copy()
    Q_prev = None
    for start, end in og.restart_windows(5, restarts):
        Xin = X0 if stale == "gram" else X   # slip: Gram matrix of the old iterate
        Q = window(Xin, rows[start:end])
        if stale == "factor" and Q_prev is not None:
            Q = Q @ Q_prev                   # slip: factor not reset at the restart
        X = Q @ X
        Q_prev = Q
    return X.T if tr else X


@pytest.mark.parametrize("slip", ["one_sided", "stale_gram", "stale_factor"])
def test_planted_slips_fail_the_pins(slip):
    G = np.random.default_rng(9).standard_normal((8, 15))
    ref = oracle.newton_schulz(G, 5)
    if slip == "one_sided":
        got = _run_with(_one_sided_r, G)
    elif slip == "stale_gram":
        got = _run_with(og.gram_window_factor, G, stale="gram")
    else:
        got = _run_with(og.gram_window_factor, G, stale="factor")
    assert _rel(got, ref) > 1e-3
    # and the unmodified routine passes the same check
    assert _rel(_run_with(og.gram_window_factor, G), ref) <= 1e-10


@pytest.mark.parametrize("restarts", [(), (2,), (1, 3)])
def test_gram_equals_direct_with_the_polar_express_table(restarts):
    """The Gram algebra holds for any table, including the Polar Express
    rows with their large first step (a ~ 8, b ~ -22, c ~ 15)."""
    from oracle import polar_express as pe
    rows = pe.polar_express_rows(5)
    for shape in [(9, 23), (23, 9), (12, 12)]:
        G = np.random.default_rng(hash((shape, restarts)) % 2**32).standard_normal(shape)
        got = og.gram_newton_schulz(G, 5, coeffs=rows, restarts=restarts)
        ref = oracle.newton_schulz(G, 5, coeffs=rows)
        assert _rel(got, ref) <= 1e-9

"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each test checks the oracle against something the pages or the mathematics
fix, chosen so that a plausible slip in the oracle (a dropped term, a wrong
sign, a reversed coefficient order, X^T X for X X^T, eps in the wrong place,
a missing transpose back) fails at least one of them.  The last test plants
each of those slips in a copy of the iteration and shows that the SVD closed
form catches it.
"""
import inspect
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import step as om


def _read_rows(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _coeffs_from_golden(golden_dir):
    return [tuple(float(v) for v in r)
            for r in _read_rows(os.path.join(golden_dir, "you_coefficients.txt"))]


def _scalar_p(sigma, rows):
    """Composed scalar quintic p_K o ... o p_1, p_k(s) = a s + b s^3 + c s^5.

    An odd matrix polynomial acts on singular values through this scalar
    map, so the NS output is U diag(p(sigma)) V^T.
    """
    s = sigma
    for a, b, c in rows:
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def _closed_form(G, rows, eps):
    """NS output from the SVD of the normalised matrix (independent route)."""
    G = np.asarray(G, np.float64)
    U, S, Vt = np.linalg.svd(G, full_matrices=False)
    nrm = math.sqrt(float(np.sum(G * G))) + eps
    sig = S / nrm
    return (U * np.array([_scalar_p(float(s), rows) for s in sig])) @ Vt


# --------------------------------------------------------------------------
# constants the pages print
# --------------------------------------------------------------------------

def test_coefficient_table_matches_printed(golden_dir):
    gold = _coeffs_from_golden(golden_dir)
    assert len(gold) == 5
    assert [tuple(r) for r in oracle.YOU_COEFFICIENTS] == gold


def test_defaults_match_printed_signature(golden_dir):
    gold = {k: float(v) for k, v in _read_rows(os.path.join(golden_dir, "muon_defaults.txt"))}
    sig = inspect.signature(om.muon_step).parameters
    assert sig["lr"].default == gold["lr"]
    assert sig["mu"].default == gold["momentum"]
    assert sig["wd"].default == gold["weight_decay"]
    assert sig["ns_steps"].default == gold["ns_steps"]
    assert bool(sig["nesterov"].default) == bool(gold["nesterov"])
    assert sig["eps"].default == gold["eps"]
    assert om.DEFAULT_EPS == gold["eps"]


def test_coefficient_rows_default_and_repeat(golden_dir):
    gold = _coeffs_from_golden(golden_dir)
    assert om.coefficient_rows(5) == gold
    assert om.coefficient_rows(3) == gold[:3]
    assert om.coefficient_rows(7) == gold + [gold[-1], gold[-1]]
    assert om.coefficient_rows(0) == []
    custom = [(3.0, -3.0, 1.0), (2.0, -1.0, 0.5)]
    assert om.coefficient_rows(2, custom) == custom
    with pytest.raises(ValueError):
        om.coefficient_rows(3, custom)
    with pytest.raises(ValueError):
        om.coefficient_rows(-1)


# --------------------------------------------------------------------------
# exact arithmetic on tiny cases
# --------------------------------------------------------------------------

def test_momentum_and_nesterov_hand_values():
    M = np.array([[1.0, 2.0]])
    G = np.array([[3.0, -1.0]])
    Mn = om.momentum_update(M, G, 0.5)
    assert np.array_equal(Mn, np.array([[3.5, 0.0]]))
    # Nesterov input uses the updated buffer: G + mu * M_new
    assert np.array_equal(om.nesterov_input(G, Mn, 0.5, True), np.array([[4.75, -1.0]]))
    assert np.array_equal(om.nesterov_input(G, Mn, 0.5, False), Mn)


def test_scalar_case_exact_rational(golden_dir):
    """1x1 matrix: every matrix product is a scalar product, so the whole
    step is a rational function of the inputs, evaluated here exactly."""
    rows = _coeffs_from_golden(golden_dir)
    g, m, w = Fraction(-3, 4), Fraction(1, 8), Fraction(1, 2)
    mu, lr, wd = Fraction(19, 20), Fraction(1, 50), Fraction(1, 10)
    eps = Fraction(1, 10 ** 7)
    m_new = mu * m + g
    u = g + mu * m_new
    x = u / (abs(u) + eps)
    for a, b, c in rows:
        a, b, c = Fraction(a), Fraction(b), Fraction(c)
        x = a * x + b * x ** 3 + c * x ** 5
    w_new = (1 - lr * wd) * w - lr * 1 * x  # scale(1,1) = 1 in mode 0
    out = om.muon_step(np.array([[float(w)]]), np.array([[float(g)]]),
                       np.array([[float(m)]]), lr=float(lr), mu=float(mu),
                       wd=float(wd), ns_steps=5, eps=float(eps))
    assert out["M"][0, 0] == pytest.approx(float(m_new), rel=1e-15)
    assert out["O"][0, 0] == pytest.approx(float(x), rel=1e-13)
    assert out["W"][0, 0] == pytest.approx(float(w_new), rel=1e-14)
    # p(1) of the printed table: the composed quintic at sigma = 1, evaluated exactly
    assert float(_scalar_p(Fraction(1), [tuple(map(Fraction, r)) for r in rows])) == pytest.approx(0.97835, abs=5e-6)


def test_zero_gradient_gives_zero_output():
    G = np.zeros((6, 9))
    assert np.array_equal(om.newton_schulz(G), np.zeros((6, 9)))
    out = om.muon_step(np.ones((6, 9)), G, np.zeros((6, 9)), lr=0.1, wd=0.5)
    assert np.allclose(out["W"], 0.95 * np.ones((6, 9)), rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(5, 9), (9, 5), (7, 7), (1, 6), (12, 3), (16, 24)])
def test_svd_closed_form(shape, golden_dir):
    rows = _coeffs_from_golden(golden_dir)
    rng = np.random.default_rng(hash(shape) % 2 ** 32)
    G = rng.standard_normal(shape)
    got = om.newton_schulz(G, 5, None, 1e-7)
    want = _closed_form(G, rows, 1e-7)
    assert np.max(np.abs(got - want)) < 1e-12


def test_svd_closed_form_custom_coefficients():
    rows = [(3.4445, -4.7750, 2.0315)] * 4 + [(1.5, -0.5, 0.0)]
    rng = np.random.default_rng(5)
    G = rng.standard_normal((8, 11))
    got = om.newton_schulz(G, 5, rows)
    assert np.max(np.abs(got - _closed_form(G, rows, 1e-7))) < 1e-12


def test_rank_one_and_eps_placement(golden_dir):
    rows = _coeffs_from_golden(golden_dir)
    rng = np.random.default_rng(11)
    u = rng.standard_normal(7); u /= np.linalg.norm(u)
    v = rng.standard_normal(4); v /= np.linalg.norm(v)
    for alpha in (3.0, 1e-7, 2.5e-8):
        G = alpha * np.outer(u, v)
        sigma = alpha / (alpha + 1e-7)   # ||G||_F = alpha, eps after the norm
        want = _scalar_p(sigma, rows) * np.outer(u, v)
        got = om.newton_schulz(G)
        assert np.max(np.abs(got - want)) < 1e-12 * max(1.0, np.max(np.abs(want)))


def test_scaled_orthogonal(golden_dir):
    rows = _coeffs_from_golden(golden_dir)
    rng = np.random.default_rng(3)
    n = 6
    Q, _ = np.linalg.qr(rng.standard_normal((n, n)))
    for alpha in (1.0, 1e-6):
        sigma = alpha / (alpha * math.sqrt(n) + 1e-7)
        got = om.newton_schulz(alpha * Q)
        assert np.max(np.abs(got - _scalar_p(sigma, rows) * Q)) < 1e-12


def test_orthogonal_equivariance():
    rng = np.random.default_rng(21)
    X = rng.standard_normal((6, 10))
    Q, _ = np.linalg.qr(rng.standard_normal((6, 6)))
    R, _ = np.linalg.qr(rng.standard_normal((10, 10)))
    lhs = om.newton_schulz(Q @ X @ R)
    rhs = Q @ om.newton_schulz(X) @ R
    assert np.max(np.abs(lhs - rhs)) < 1e-12


def test_transpose_symmetry():
    rng = np.random.default_rng(8)
    G = rng.standard_normal((13, 5))      # tall: oracle transposes
    a = om.newton_schulz(G)
    b = om.newton_schulz(G.T.copy())      # wide: no transpose
    assert a.shape == G.shape
    assert np.max(np.abs(a - b.T)) < 1e-13


def test_orientation_rule():
    tall = np.arange(12.0).reshape(4, 3)
    Y, t = om.orient(tall)
    assert t and Y.shape == (3, 4)
    Y, t = om.orient(tall.T)
    assert not t and Y.shape == (3, 4)
    Y, t = om.orient(np.eye(3))
    assert not t


def test_update_scale_and_apply_hand_values():
    assert om.update_scale(512, 128, 0) == 2.0
    assert om.update_scale(128, 512, 0) == 1.0
    assert om.update_scale(4096, 4096, 0) == 1.0
    assert om.update_scale(14336, 4096, 1) == 1.0
    assert om.update_scale(4096, 1024, 2) == pytest.approx(12.8, rel=1e-15)
    W = np.array([[1.0, -2.0]])
    O = np.array([[0.5, 0.25]])
    got = om.apply_update(W, O, lr=0.1, wd=0.5, scale=2.0)
    assert np.allclose(got, [[0.95 - 0.1, -1.9 - 0.05]], rtol=0, atol=1e-15)


def test_muon_step_composes_the_steps(golden_dir):
    """muon_step equals the closed-form route assembled step by step."""
    rows = _coeffs_from_golden(golden_dir)
    rng = np.random.default_rng(4)
    W = rng.standard_normal((9, 4)); G = rng.standard_normal((9, 4)); M = rng.standard_normal((9, 4))
    out = om.muon_step(W, G, M, lr=0.03, mu=0.9, wd=0.1, ns_steps=5)
    M_new = 0.9 * M + G
    U = G + 0.9 * M_new
    O = _closed_form(U, rows, 1e-7)
    W_new = (1 - 0.03 * 0.1) * W - 0.03 * 1.5 * O     # scale sqrt(9/4) = 1.5
    assert np.max(np.abs(out["M"] - M_new)) < 1e-15
    assert np.max(np.abs(out["O"] - O)) < 1e-12
    assert np.max(np.abs(out["W"] - W_new)) < 1e-12
    assert out["scale"] == 1.5


# --------------------------------------------------------------------------
# planted mistakes: the closed form must reject each slip
# --------------------------------------------------------------------------

def _mutant_ns(G, rows, eps, slip):
    G = np.asarray(G, np.float64)
    t = G.shape[0] > G.shape[1]
    Y = G.T if t else G
    if slip == "eps_inside_sqrt":
        X = Y / np.sqrt(np.sum(Y * Y) + eps)
    else:
        X = Y / (np.sqrt(np.sum(Y * Y)) + eps)
    seq = list(reversed(rows)) if slip == "reversed_rows" else rows
    for a, b, c in seq:
        A = (X.T @ X) if slip == "gram_transposed" else (X @ X.T)
        if slip == "drop_c":
            B = b * A
        elif slip == "flip_b":
            B = -b * A + c * (A @ A)
        else:
            B = b * A + c * (A @ A)
        X = a * X + B @ X
    if slip == "no_transpose_back":
        return X
    return X.T if t else X


@pytest.mark.parametrize("slip", ["drop_c", "flip_b", "reversed_rows",
                                  "gram_transposed", "eps_inside_sqrt",
                                  "no_transpose_back"])
def test_planted_slips_are_caught(slip, golden_dir):
    rows = _coeffs_from_golden(golden_dir)
    rng = np.random.default_rng(2)
    if slip == "eps_inside_sqrt":
        G = 1e-7 * rng.standard_normal((6, 6)) / 6.0   # norm near eps
    elif slip == "no_transpose_back":
        G = rng.standard_normal((6, 6))
        G = G + G.T                                      # symmetric: shape hides nothing
        G = np.vstack([G, rng.standard_normal((1, 6))])  # then make it tall
    else:
        G = rng.standard_normal((6, 6))
    want = _closed_form(G, rows, 1e-7)
    assert np.max(np.abs(om.newton_schulz(G) - want)) < 1e-12
    with np.errstate(all="ignore"):
        bad = _mutant_ns(G, rows, 1e-7, slip)
    if bad.shape != want.shape:
        return  # shape mismatch already fails any comparison
    close = bool(np.all(np.isfinite(bad))) and float(np.max(np.abs(bad - want))) <= 1e-3
    assert not close

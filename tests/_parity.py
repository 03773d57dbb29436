"""Shared parity checks of the GPU tests.

The momentum bar is element by element: the GPU updates each element with
one fused multiply-add of fp32 values, a single rounding of the exact
``mu * M + G``, so every element sits within 2^-24 of the fp64 oracle's value
relative to itself (an exact zero stays zero).  The bar, 1e-6 relative per
element, leaves room for nothing else; the Frobenius ratio is reported
beside it.
"""
import numpy as np

MOM_TOL = 1e-6


def rel_fro(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    nr = np.linalg.norm(ref)
    return np.linalg.norm(got - ref) / nr if nr > 0 else np.linalg.norm(got - ref)


def assert_momentum(got, ref, what=""):
    """Every element of the GPU momentum within MOM_TOL of the oracle's,
    relative to the oracle's element."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape
    err = np.abs(got - ref)
    bad = err > MOM_TOL * np.abs(ref)
    if bad.any():
        i = np.unravel_index(int(np.argmax(np.where(bad, err / np.maximum(np.abs(ref), 1e-300), 0))), ref.shape)
        raise AssertionError("momentum %s: %d elements past %.0e relative, worst at %s: got %r, oracle %r "
                             "(Frobenius ratio %.2e)" % (what, int(bad.sum()), MOM_TOL, i, got[i], ref[i],
                                                         rel_fro(got, ref)))


def spectrum_matrix(rows, cols, ratio, seed):
    """Seeded fp32 rows x cols matrix U diag(sv) V^T with orthonormal U, V
    (QR of Gaussians) and singular values spread log-uniformly over
    [1/ratio, 1]: an input of condition number about ``ratio``."""
    rng = np.random.default_rng(seed)
    m = min(rows, cols)
    u, _ = np.linalg.qr(rng.standard_normal((rows, m)))
    v, _ = np.linalg.qr(rng.standard_normal((cols, m)))
    sv = np.exp(rng.uniform(np.log(1.0 / ratio), 0.0, m))
    return np.ascontiguousarray((u * sv) @ v.T, dtype=np.float32)

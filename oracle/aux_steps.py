"""fp64 oracle of the two other parts of ``Muon.step`` built here: AdamW on the
non-Muon parameters and (segmented) gradient-norm clipping of Muon gradients.

Test infrastructure only (tests/, the smoke check and bench.py's CPU legs);
it shares nothing with the CUDA library.

AdamW -- DMuon "API Reference", section *Muon*: symmetric (non-dedicated)
parameters are updated with AdamW, defaults ``adamw_lr=1e-3``,
``adamw_betas=(0.9, 0.999)``, ``adamw_weight_decay=0.01``,
``adamw_eps=1e-8``.  The pages name the optimizer but print no formula;
reading: the standard decoupled-weight-decay Adam with bias correction
(Loshchilov and Hutter), the form PyTorch's ``torch.optim.AdamW`` uses:

    p <- p * (1 - lr*wd)
    m <- b1*m + (1 - b1)*g ;  v <- b2*v + (1 - b2)*g^2
    p <- p - lr * (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps)

Clipping -- DMuon "API Reference", sections *clip_grad_norm_* (global norm
over the Muon gradients, statistics ``total_norm`` before clipping,
``clip_coef``, ``clipped``, ``found_inf``; ``max_norm=None`` only reports)
and *clip_grad_norm_buckets_* (each bucket keeps its own norm and clip
coefficient).  Reading: the coefficient is ``max_norm / (total_norm + 1e-6)``
and gradients are scaled only when it is below 1, as in PyTorch's
``clip_grad_norm_``.
"""
import numpy as np

ADAMW_DEFAULTS = {"lr": 1e-3, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8, "weight_decay": 0.01}
CLIP_EPS = 1e-6


def adamw_step(p, g, m, v, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01):
    """One AdamW step on one tensor; ``step`` is the 1-based step count.
    Returns (p, m, v) in float64."""
    p = np.asarray(p, np.float64) * (1.0 - lr * weight_decay)
    g = np.asarray(g, np.float64)
    m = beta1 * np.asarray(m, np.float64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(v, np.float64) + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** step)
    v_hat = v / (1.0 - beta2 ** step)
    p = p - lr * m_hat / (np.sqrt(v_hat) + eps)
    return p, m, v


def bucket_norms(grads, buckets, n_buckets):
    """Euclidean norm of the concatenation of each bucket's gradients."""
    sq = [0.0] * n_buckets
    for g, b in zip(grads, buckets):
        a = np.asarray(g, np.float64)
        sq[b] += float(np.sum(a * a))
    return [float(np.sqrt(s)) for s in sq]


def clip_coefficients(norms, max_norm):
    """``max_norm / (norm + 1e-6)`` per bucket (None when only reporting)."""
    if max_norm is None:
        return [None] * len(norms)
    return [max_norm / (n + CLIP_EPS) for n in norms]


def clip_grad_norm_buckets(grads, buckets, n_buckets, max_norm):
    """Segmented clipping.  Returns (clipped grads as float64 arrays,
    per-bucket norms, per-bucket coefficients, per-bucket found_inf)."""
    norms = bucket_norms(grads, buckets, n_buckets)
    coefs = clip_coefficients(norms, max_norm)
    out = []
    for g, b in zip(grads, buckets):
        a = np.asarray(g, np.float64)
        c = coefs[b]
        out.append(a * c if (c is not None and c < 1.0) else a.copy())
    found_inf = [not np.isfinite(n) for n in norms]
    return out, norms, coefs, found_inf

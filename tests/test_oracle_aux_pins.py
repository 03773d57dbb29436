"""Pins of the AdamW and clipping oracles (CPU only).

Each is checked against hand-computed values and against the PyTorch
routine that implements the same textbook definition, run in float64.
"""
import math

import numpy as np
import pytest

from oracle import aux_steps as ox

torch = pytest.importorskip("torch")


def test_adamw_defaults_match_printed_signature():
    # DMuon "API Reference", Muon signature: adamw_lr, adamw_betas, adamw_weight_decay, adamw_eps
    assert ox.ADAMW_DEFAULTS == {"lr": 1e-3, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8,
                                 "weight_decay": 0.01}


def test_adamw_first_step_hand_values():
    # step 1 from zero moments: m_hat = g, v_hat = g^2, so the update is
    # lr * g / (|g| + eps) after the decoupled decay
    p, g = np.array([1.0, -2.0, 0.5]), np.array([0.3, -0.4, 0.0])
    lr, wd, eps = 0.1, 0.5, 1e-8
    p2, m, v = ox.adamw_step(p, g, np.zeros(3), np.zeros(3), 1, lr=lr, weight_decay=wd, eps=eps)
    want = p * (1 - lr * wd) - lr * g / (np.abs(g) + eps)
    assert np.allclose(p2, want, rtol=0, atol=1e-15)
    assert np.allclose(m, 0.1 * g) and np.allclose(v, 0.001 * g * g)


def test_adamw_matches_torch_over_steps():
    rng = np.random.default_rng(0)
    p0 = rng.standard_normal((5, 7))
    tp = torch.nn.Parameter(torch.tensor(p0, dtype=torch.float64))
    opt = torch.optim.AdamW([tp], lr=3e-3, betas=(0.8, 0.95), eps=1e-6, weight_decay=0.1)
    p, m, v = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
    for step in range(1, 6):
        g = rng.standard_normal((5, 7))
        tp.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        p, m, v = ox.adamw_step(p, g, m, v, step, lr=3e-3, beta1=0.8, beta2=0.95, eps=1e-6,
                                weight_decay=0.1)
    assert np.max(np.abs(p - tp.detach().numpy())) < 1e-13


def test_clip_hand_values():
    grads = [np.array([3.0]), np.array([4.0]), np.array([1.0, 1.0])]
    out, norms, coefs, inf = ox.clip_grad_norm_buckets(grads, [0, 0, 1], 2, 1.0)
    assert norms[0] == 5.0 and norms[1] == pytest.approx(math.sqrt(2.0), rel=1e-15)
    assert coefs[0] == pytest.approx(1.0 / (5.0 + 1e-6), rel=1e-15)
    assert np.allclose(out[0], 3.0 / (5.0 + 1e-6)) and np.allclose(out[1], 4.0 / (5.0 + 1e-6))
    assert np.allclose(out[2], 1.0 / (math.sqrt(2.0) + 1e-6))
    assert inf == [False, False]
    # below the limit nothing changes; statistics-only leaves gradients alone
    out2, _, coefs2, _ = ox.clip_grad_norm_buckets(grads, [0, 0, 1], 2, 10.0)
    assert coefs2[0] > 1 and np.array_equal(out2[0], grads[0])
    out3, norms3, coefs3, _ = ox.clip_grad_norm_buckets(grads, [0, 0, 1], 2, None)
    assert coefs3 == [None, None] and np.array_equal(out3[2], grads[2]) and norms3 == norms


def test_clip_matches_torch_per_bucket():
    rng = np.random.default_rng(1)
    grads = [rng.standard_normal(s) for s in ((4, 6), (10,), (3, 3), (8, 2))]
    buckets = [0, 1, 0, 1]
    out, norms, _, _ = ox.clip_grad_norm_buckets(grads, buckets, 2, 0.7)
    for b in range(2):
        ps = [torch.nn.Parameter(torch.zeros(g.shape, dtype=torch.float64))
              for g, bb in zip(grads, buckets) if bb == b]
        for p, g in zip(ps, [g for g, bb in zip(grads, buckets) if bb == b]):
            p.grad = torch.tensor(g, dtype=torch.float64)
        tn = torch.nn.utils.clip_grad_norm_(ps, 0.7)
        assert float(tn) == pytest.approx(norms[b], rel=1e-14)
        mine = [o for o, bb in zip(out, buckets) if bb == b]
        for p, o in zip(ps, mine):
            assert np.max(np.abs(p.grad.numpy() - o)) < 1e-15


def test_clip_found_inf():
    _, norms, _, inf = ox.clip_grad_norm_buckets([np.array([1.0, np.inf]), np.array([2.0])],
                                                 [0, 1], 2, 1.0)
    assert inf == [True, False] and math.isinf(norms[0])

"""GPU parity of the AdamW and segmented-clipping kernels against the fp64
oracle (oracle/aux_steps.py), through the C ABI.

Bars: AdamW moments within 1e-6 relative Frobenius error; parameters
elementwise within 16 * steps * 2^-24 * max(|p|, 1) of the oracle (each step
rounds p a few times in fp32: the decay product, the quotient, the fused
update), and the accumulated update p' - p within 1e-5 relative Frobenius
error with lr = 0.1, where the update (~0.1 per step) dominates the rounding
of p; clipping norms and coefficients within 1e-6 relative, clipped
gradients within 1e-6 relative Frobenius.
Sizes cover several 8192-element tiles, ragged tails (numel % 4 != 0) and
tensors only 4-byte aligned (scalar path).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import newton_schulz_nesterov_gb300 as dm  # noqa: E402
from newton_schulz_nesterov_gb300 import _build  # noqa: E402
from oracle import aux_steps as ox  # noqa: E402

pytestmark = pytest.mark.gpu

SIZES = [(1,), (7,), (4096,), (8193,), (3, 5), (129, 257), (64, 8192), (1000, 37)]


def rel(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    nr = np.linalg.norm(ref)
    return np.linalg.norm(got - ref) / nr if nr > 0 else np.linalg.norm(got - ref)


@pytest.fixture(scope="module")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    h = dm.Handle(0)
    yield h
    h.close()


def _unaligned(t):
    """Same values in a buffer shifted by one float: 4-byte but not 16-byte aligned."""
    buf = torch.empty(t.numel() + 1, device="cuda")
    v = buf[1:].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("unaligned", [False, True])
def test_adamw_three_steps(handle, unaligned):
    gen = torch.Generator().manual_seed(31)
    P = [torch.randn(s, generator=gen) for s in SIZES]
    M = [torch.zeros(s) for s in SIZES]
    V = [torch.zeros(s) for s in SIZES]
    dev = lambda ts: [(_unaligned(t.cuda()) if unaligned else t.clone().cuda()) for t in ts]  # noqa: E731
    Pd, Md, Vd = dev(P), dev(M), dev(V)
    Pr = [p.numpy().astype(np.float64) for p in P]
    Mr = [np.zeros(s) for s in SIZES]
    Vr = [np.zeros(s) for s in SIZES]
    hp = dict(lr=0.1, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    f32 = {k: float(np.float32(v)) for k, v in hp.items()}
    for step in range(1, 4):
        G = [torch.randn(s, generator=gen) for s in SIZES]
        Gd = dev(G)
        dm.dmuon_adamw_step(handle.h, Pd, Gd, Md, Vd, step=step, **hp)
        for i in range(len(SIZES)):
            Pr[i], Mr[i], Vr[i] = ox.adamw_step(Pr[i], G[i].numpy(), Mr[i], Vr[i], step, **f32)
    assert handle.status()[0] == 0
    for i in range(len(SIZES)):
        p0 = P[i].numpy().astype(np.float64)
        assert rel(Md[i].cpu().numpy(), Mr[i]) <= 1e-6, ("m", SIZES[i])
        assert rel(Vd[i].cpu().numpy(), Vr[i]) <= 1e-6, ("v", SIZES[i])
        pg = Pd[i].cpu().numpy().astype(np.float64)
        bound = 16 * 3 * 2.0 ** -24 * np.maximum(np.abs(Pr[i]), 1.0)
        assert np.all(np.abs(pg - Pr[i]) <= bound), ("p elementwise", SIZES[i])
        assert rel(pg - p0, Pr[i] - p0) <= 1e-5, ("p update", SIZES[i])


def test_adamw_argument_errors(handle):
    x = torch.zeros(8, device="cuda")
    y, z, w = torch.zeros_like(x), torch.zeros_like(x), torch.zeros_like(x)
    call = lambda **k: dm.dmuon_adamw_step_ptrs(handle.h, [x.data_ptr()], [k.get("g", y.data_ptr())],  # noqa: E731
                                                [z.data_ptr()], [w.data_ptr()], [k.get("n", 8)],
                                                step=k.get("step", 1), beta1=k.get("b1", 0.9),
                                                check=False)
    assert call(step=0) == -1
    assert call(b1=1.0) == -1
    assert call(n=0) == -1
    assert call(g=x.data_ptr()) == -1          # aliasing params
    assert call(g=y.data_ptr() + 2) == -2      # not 4-byte aligned
    assert call() == 0


@pytest.mark.parametrize("unaligned", [False, True])
def test_clip_segmented(handle, unaligned):
    gen = torch.Generator().manual_seed(37)
    G = [torch.randn(s, generator=gen) * (i + 1) for i, s in enumerate(SIZES)]
    buckets = [0, 1, 2, 0, 1, 2, 0, 1]
    dev = lambda ts: [(_unaligned(t.cuda()) if unaligned else t.clone().cuda()) for t in ts]  # noqa: E731
    for max_norm in (5.0, 1e9, 0.0):
        Gd = dev(G)
        norms, coefs = dm.dmuon_clip_grad_norm(handle.h, Gd, max_norm, buckets, 3)
        out, rn, rc_, _ = ox.clip_grad_norm_buckets([g.numpy() for g in G], buckets, 3,
                                                    max_norm if max_norm > 0 else None)
        for b in range(3):
            assert abs(norms[b] - rn[b]) <= 1e-6 * rn[b]
            if max_norm > 0:
                assert abs(coefs[b] - rc_[b]) <= 1e-6 * rc_[b]
            else:
                assert coefs[b] == -1.0
        for i in range(len(SIZES)):
            got = Gd[i].cpu().numpy()
            if max_norm > 0:
                assert rel(got, out[i]) <= 1e-6, (max_norm, SIZES[i])
            else:
                assert np.array_equal(got, G[i].numpy())   # statistics only: untouched


def test_clip_global_and_found_inf(handle):
    G = [torch.full((100,), 3.0, device="cuda"), torch.full((44,), 4.0, device="cuda")]
    norms, coefs = dm.dmuon_clip_grad_norm(handle.h, G, 1.0)
    want = float(np.sqrt(100 * 9.0 + 44 * 16.0))
    assert abs(norms[0] - want) <= 1e-6 * want
    assert abs(float(G[0][0]) - 3.0 / (want + 1e-6)) <= 1e-6
    H = [torch.ones(16, device="cuda"), torch.ones(16, device="cuda")]
    H[1][3] = float("inf")
    norms, _ = dm.dmuon_clip_grad_norm(handle.h, H, 1.0, [0, 1], 2)
    assert np.isfinite(norms[0]) and not np.isfinite(norms[1])

"""GPU parity of the fused small-matrix kernel (oriented m <= 128, n <= 512,
one CTA per matrix) against the fp64 oracle, and its integration with the
chunked tensor-core path in one call: mixed lists (the small matrices run
in plan order after the large ones, so pointer sets and flags are permuted
and must come back in the caller's order), every step option, the wait
limit, and the profile/launch accounting.

Bars as in the other parity tests: momentum <= 1e-6 relative Frobenius
error, update and NS output <= 3e-2.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import newton_schulz_nesterov_gb300 as dm  # noqa: E402
from newton_schulz_nesterov_gb300 import _build, workloads  # noqa: E402
import oracle  # noqa: E402

from _parity import assert_momentum  # noqa: E402

pytestmark = pytest.mark.gpu

NS_TOL = 3e-2
F32 = lambda x: float(np.float32(x))  # noqa: E731

# every small-kernel shape class: 1-wide, ragged, exactly one tile, both
# orientations, the 512-column limit, square
SMALL = [(1, 1), (1, 37), (37, 1), (3, 5), (5, 3), (64, 256), (256, 64), (128, 512),
         (512, 128), (128, 128), (100, 500), (500, 100), (33, 129), (127, 65), (7, 300),
         (65, 65), (2, 512), (512, 1)]


def rel_fro(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    nr = np.linalg.norm(ref)
    d = np.linalg.norm(got - ref)
    return d / nr if nr > 0 else d


@pytest.fixture(scope="module")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    h = dm.Handle(0)
    yield h
    h.close()


def _dev(ts):
    return [t.clone().cuda() for t in ts]


def _inputs(shapes, seed):
    gen = torch.Generator().manual_seed(seed)
    Ws = [torch.rand(s, generator=gen) - 0.5 for s in shapes]
    Gs = [torch.randn(s, generator=gen) for s in shapes]
    Ms = [torch.randn(s, generator=gen) for s in shapes]
    return Ws, Gs, Ms


def _check_step(h, shapes, seed, lr=0.05, mu=0.9, ns_steps=5, wd=0.0, nesterov=True, scale_mode=0,
                coeffs=None):
    Ws, Gs, Ms = _inputs(shapes, seed)
    Wd, Gd, Md = _dev(Ws), _dev(Gs), _dev(Ms)
    h.step(Wd, Gd, Md, lr=lr, mu=mu, ns_steps=ns_steps, weight_decay=wd, nesterov=nesterov,
           scale_mode=scale_mode, coeffs=coeffs)
    rc, flags = h.status(len(shapes))
    assert rc == 0 and not any(flags)
    for i, s in enumerate(shapes):
        ref = oracle.muon_step(Ws[i].numpy(), Gs[i].numpy(), Ms[i].numpy(), lr=F32(lr), mu=F32(mu),
                               wd=F32(wd), ns_steps=ns_steps, coeffs=coeffs, nesterov=nesterov,
                               scale_mode=scale_mode)
        W0 = Ws[i].numpy().astype(np.float64)
        assert_momentum(Md[i].cpu().numpy(), ref["M"], str(s))
        e = rel_fro(Wd[i].cpu().numpy().astype(np.float64) - W0, ref["W"] - W0)
        assert e <= NS_TOL, ("update", s, e)
    return Wd, Md


def test_small_shapes_step(handle):
    _check_step(handle, SMALL, 101)
    assert "small-matrix kernel %d;" % len(SMALL) in dm.dmuon_plan_summary(handle.h)


def test_small_shapes_newton_schulz(handle):
    gen = torch.Generator().manual_seed(103)
    ins = [torch.randn(s, generator=gen) for s in SMALL]
    outs = [torch.empty(s, device="cuda") for s in SMALL]
    handle.newton_schulz(_dev(ins), outs)
    assert handle.status()[0] == 0
    for x, o, s in zip(ins, outs, SMALL):
        e = rel_fro(o.cpu().numpy(), oracle.newton_schulz(x.numpy()))
        assert e <= NS_TOL, (s, e)


@pytest.mark.parametrize("kw", [
    dict(ns_steps=0), dict(ns_steps=1), dict(ns_steps=2), dict(ns_steps=7),
    dict(nesterov=False), dict(wd=0.1), dict(scale_mode=1), dict(scale_mode=2),
    dict(ns_steps=3, coeffs=[(3.0, -3.2, 1.2), (2.5, -2.0, 0.5), (1.875, -1.25, 0.375)]),
])
def test_small_step_options(handle, kw):
    _check_step(handle, [(96, 300), (300, 96), (128, 512), (5, 3)], 107, **kw)


def test_newton_schulz_zero_steps_is_the_normalised_input(handle):
    """ns_steps = 0: O = G / (||G||_F + eps), exactly in fp32 terms."""
    gen = torch.Generator().manual_seed(109)
    shapes = [(64, 256), (300, 17)]
    ins = [torch.randn(s, generator=gen) for s in shapes]
    outs = [torch.empty(s, device="cuda") for s in shapes]
    handle.newton_schulz(_dev(ins), outs, ns_steps=0)
    assert handle.status()[0] == 0
    for x, o in zip(ins, outs):
        ref = x.numpy().astype(np.float64) / (np.linalg.norm(x.numpy().astype(np.float64)) + 1e-7)
        assert rel_fro(o.cpu().numpy(), ref) <= 1e-6


def test_small_scaled_inputs(handle):
    """The kernel takes max |U| first and prescales X0 = p U by the power of
    two that puts it near 2^10, and rescales the iterate when ||U|| is far
    below eps: inputs over the whole fp32 range meet the bar."""
    gen = torch.Generator().manual_seed(131)
    shapes = [(64, 256), (512, 128), (37, 300)]
    base = [torch.randn(s, generator=gen) for s in shapes]
    for scale in (1e-30, 1e-20, 1e-6, 1.0, 1e3, 1e15, 1e30):
        ins = [(b * scale).cuda() for b in base]
        outs = [torch.empty_like(x) for x in ins]
        handle.newton_schulz(ins, outs)
        assert handle.status()[0] == 0
        assert "small-matrix kernel %d;" % len(shapes) in dm.dmuon_plan_summary(handle.h)
        for x, o, sh in zip(ins, outs, shapes):
            assert bool(torch.isfinite(o).all()), (scale, sh)
            e = rel_fro(o.cpu().numpy(), oracle.newton_schulz(x.cpu().numpy().astype(np.float64)))
            assert e <= NS_TOL, (scale, sh, e)


@pytest.mark.parametrize("ratio", [1e2, 1e4])
def test_small_ill_conditioned_inputs(handle, ratio):
    """Singular values spread log-uniformly over [1/ratio, 1] on the small
    kernel, with the printed and the Polar Express tables."""
    from _parity import spectrum_matrix
    from oracle import polar_express as pe
    shapes = [(128, 512), (512, 128), (100, 100), (64, 256)]
    ins = [torch.from_numpy(spectrum_matrix(r, c, ratio, 133 + k)) for k, (r, c) in enumerate(shapes)]
    for coeffs, ref_coeffs in ((None, None), (dm.dmuon_polar_express_coefficients(5), pe.polar_express_rows(5))):
        outs = [torch.empty(s, device="cuda") for s in shapes]
        handle.newton_schulz([x.cuda() for x in ins], outs, coeffs=coeffs)
        assert handle.status()[0] == 0
        for x, o, sh in zip(ins, outs, shapes):
            e = rel_fro(o.cpu().numpy(), oracle.newton_schulz(x.numpy().astype(np.float64), 5, coeffs=ref_coeffs))
            assert e <= NS_TOL, (sh, ratio, coeffs is None, e)


def test_mixed_list_keeps_caller_order(handle):
    """Large and small matrices interleaved: each gets its own buffers'
    result (the device pointer set is permuted into plan order)."""
    shapes = [(300, 500), (64, 256), (700, 300), (5, 3), (257, 257), (128, 512), (1, 1), (200, 640)]
    _check_step(handle, shapes, 113)
    summary = dm.dmuon_plan_summary(handle.h)
    assert "small-matrix kernel 4;" in summary and "matrices 8" in summary


def test_mixed_list_nonfinite_flags_in_caller_order(handle):
    shapes = [(300, 500), (64, 96), (700, 300), (96, 64)]
    Ws = [torch.zeros(s, device="cuda") for s in shapes]
    Gs = [torch.ones(s, device="cuda") for s in shapes]
    Ms = [torch.zeros(s, device="cuda") for s in shapes]
    Gs[3][5, 7] = float("nan")
    Gs[2][1, 1] = float("inf")
    handle.step(Ws, Gs, Ms)
    rc, flags = handle.status(4)
    assert rc == -5 and flags == [0, 0, 1, 1]
    assert handle.status(4) == (0, [0, 0, 0, 0])


def test_small_path_off_matches_on(handle):
    """The same list with the small kernel on and off: both meet the oracle
    bar, and they agree with each other to fp16 rounding."""
    shapes = [(64, 256), (256, 64), (128, 512), (33, 129), (3, 5)]
    res = []
    for on in (True, False):
        with dm.Handle(0) as h2:
            dm.dmuon_set_small_path(h2.h, on)
            Wd, Md = _check_step(h2, shapes, 127)
            n_small = len(shapes) if on else 0
            assert "small-matrix kernel %d;" % n_small in dm.dmuon_plan_summary(h2.h)
            res.append(([w.cpu() for w in Wd], [m.cpu() for m in Md]))
    for a, b in zip(res[0][1], res[1][1]):
        assert torch.equal(a, b)            # momentum: same fp32 fused multiply-adds
    Ws, _, _ = _inputs(shapes, 127)
    for a, b, w0 in zip(res[0][0], res[1][0], Ws):
        assert rel_fro((a - w0).numpy(), (b - w0).numpy()) <= 2e-2


def test_small_kernel_deterministic(handle):
    shapes = [(128, 512), (512, 128), (64, 256), (1, 37)]
    Ws, Gs, Ms = _inputs(shapes, 131)
    Gd = _dev(Gs)
    res = []
    for _ in range(2):
        Wd, Md = _dev(Ws), _dev(Ms)
        handle.step(Wd, Gd, Md)
        torch.cuda.synchronize()
        res.append([x.cpu() for x in Wd + Md])
    for a, b in zip(*res):
        assert torch.equal(a, b)


def test_small_launch_count_and_profile(handle):
    """A list of small matrices is one launch, whatever ns_steps is."""
    w = workloads.get("tinymlp_d128")
    n = len(w.shapes)
    Wd = [workloads.weight(w, i, "cuda") for i in range(n)]
    Gd = [workloads.grad(w, i, 0, "cuda") for i in range(n)]
    Md = [workloads.momentum(w, i, "cuda") for i in range(n)]
    dm.dmuon_profile_enable(handle.h, True)
    dm.dmuon_profile_read(handle.h)
    for ns in (5, 0):
        before = dm.dmuon_launch_count(handle.h)
        handle.step(Wd, Gd, Md, ns_steps=ns)
        assert dm.dmuon_launch_count(handle.h) - before == 1
    prof = dm.dmuon_profile_read(handle.h)
    dm.dmuon_profile_enable(handle.h, False)
    assert prof["small"][1] == 2 and prof["momentum"][1] == 0 and prof["gram"][1] == 0
    assert handle.status()[0] == 0


def test_small_wait_timeout_is_reported_and_context_recovers(handle):
    """A 1 ns wait limit: each CTA's first product wait gives up, the CTAs
    agree, drain the issued MMAs (bounded), free tensor memory and return;
    the host reads DMUON_ERR_TIMEOUT and the next step is correct."""
    shapes = [(64, 256), (128, 512)]
    Ws, Gs, Ms = _inputs(shapes, 137)
    dm.dmuon_set_wait_timeout(handle.h, 1)
    try:
        handle.step(_dev(Ws), _dev(Gs), _dev(Ms))
        rc, _ = handle.status(2)
    finally:
        dm.dmuon_set_wait_timeout(handle.h, 0)
    assert rc == -6
    assert handle.status(2)[0] == 0
    _check_step(handle, shapes, 137)


def test_small_step_in_cuda_graph(handle):
    """Mixed list recorded in a CUDA graph: replays equal eager steps."""
    shapes = [(300, 500), (64, 256), (5, 3), (128, 512)]
    Ws, Gs, Ms = _inputs(shapes, 139)
    Wa, Ga, Ma = _dev(Ws), _dev(Gs), _dev(Ms)
    for _ in range(3):
        handle.step(Wa, Ga, Ma)
    torch.cuda.synchronize()
    with dm.Handle(0) as h2:
        Wb, Gb, Mb = _dev(Ws), _dev(Gs), _dev(Ms)
        h2.step(Wb, Gb, Mb)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            h2.step(Wb, Gb, Mb)
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        assert h2.status()[0] == 0
        for a, b in zip(Wa + Ma, Wb + Mb):
            assert torch.equal(a, b)


@pytest.mark.slow
def test_tp_70b_mixed_small_matrices_full_size(handle):
    """The 28672x8192 matrix and 512 packed 64x256 matrices in one call;
    sampled small ones against the oracle."""
    w = workloads.get("tp_70b_mixed")
    n = len(w.shapes)
    Wd = [workloads.weight(w, i, "cuda") for i in range(n)]
    Md = [workloads.momentum(w, i, "cuda") for i in range(n)]
    Gd = [workloads.grad(w, i, 0, "cuda") for i in range(n)]
    sample = [1, 2, 77, 300, 511, 512]
    W0 = {i: Wd[i].cpu() for i in sample}
    M0 = {i: Md[i].cpu() for i in sample}
    handle.step(Wd, Gd, Md)
    assert handle.status()[0] == 0
    assert "small-matrix kernel 512;" in dm.dmuon_plan_summary(handle.h)
    for i in sample:
        ref = oracle.muon_step(W0[i].numpy(), Gd[i].cpu().numpy(), M0[i].numpy(), lr=F32(0.02), mu=F32(0.95))
        w0 = W0[i].numpy().astype(np.float64)
        assert_momentum(Md[i].cpu().numpy(), ref["M"])
        assert rel_fro(Wd[i].cpu().numpy().astype(np.float64) - w0, ref["W"] - w0) <= NS_TOL, i
    del Wd, Md, Gd
    torch.cuda.empty_cache()

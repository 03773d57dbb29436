"""GPU parity of the Gram-space Newton-Schulz backend (CTA-pair fp16
Gram-window kernels + the direct Apply kernel for Q X) against the fp64 Gram
oracle (``oracle/gram.py``, itself pinned to the direct oracle and the SVD
closed form).

Bars as in the direct parity tests: NS output and weight update within 3e-2
relative Frobenius error per matrix, momentum within 1e-6.  The small-matrix
kernel (which always runs the direct iteration) is switched off on the
handles here so that small shapes exercise the Gram kernels too.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import newton_schulz_nesterov_gb300 as dm  # noqa: E402
from newton_schulz_nesterov_gb300 import _build, workloads  # noqa: E402
import oracle  # noqa: E402
from oracle import gram as og  # noqa: E402

from _parity import assert_momentum  # noqa: E402

pytestmark = pytest.mark.gpu

NS_TOL = 3e-2
F32 = lambda x: float(np.float32(x))  # noqa: E731

RAGGED = [(1, 1), (1, 37), (37, 1), (3, 5), (64, 256), (256, 64), (128, 512), (129, 257), (300, 700),
          (700, 300), (200, 200), (513, 1000), (1000, 513), (255, 2050), (8, 4100), (384, 384), (640, 96)]


def rel_fro(got, ref):
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
    dm.dmuon_set_small_path(h.h, False)
    yield h
    h.close()


def _dev(ts):
    return [t.clone().cuda() for t in ts]


def _inputs(shapes, seed):
    gen = torch.Generator().manual_seed(seed)
    return ([torch.rand(s, generator=gen) - 0.5 for s in shapes], [torch.randn(s, generator=gen) for s in shapes],
            [torch.randn(s, generator=gen) for s in shapes])


def test_gram_newton_schulz_ragged(handle):
    gen = torch.Generator().manual_seed(201)
    ins = [torch.randn(s, generator=gen) for s in RAGGED]
    outs = [torch.empty(s, device="cuda") for s in RAGGED]
    handle.gram_newton_schulz(_dev(ins), outs)
    assert handle.status()[0] == 0
    assert "backend gram" in dm.dmuon_plan_summary(handle.h)
    for x, o, s in zip(ins, outs, RAGGED):
        e = rel_fro(o.cpu().numpy(), og.gram_newton_schulz(x.numpy()))
        assert e <= NS_TOL, (s, e)


@pytest.mark.parametrize("ns_steps,restarts,coeffs", [
    (5, (), None), (5, (1,), None), (5, (1, 3), None), (5, (1, 2, 3, 4), None), (1, (2,), None),
    (3, (2,), [(3.0, -3.2, 1.2), (2.5, -2.0, 0.5), (1.875, -1.25, 0.375)]), (7, (2, 4), None), (0, (2,), None),
])
def test_gram_restart_sets(handle, ns_steps, restarts, coeffs):
    gen = torch.Generator().manual_seed(203)
    shapes = [(300, 900), (900, 300), (256, 256), (100, 2000)]
    ins = [torch.randn(s, generator=gen) for s in shapes]
    outs = [torch.empty(s, device="cuda") for s in shapes]
    handle.gram_newton_schulz(_dev(ins), outs, ns_steps=ns_steps, coeffs=coeffs, restarts=restarts)
    assert handle.status()[0] == 0
    for x, o, s in zip(ins, outs, shapes):
        ref = og.gram_newton_schulz(x.numpy(), ns_steps, coeffs=coeffs, restarts=restarts)
        e = rel_fro(o.cpu().numpy(), ref)
        assert e <= NS_TOL, (s, ns_steps, restarts, e)


def test_gram_scaled_inputs(handle):
    """Inputs over the whole fp32 range (1e-30 ... 1e30), one call per scale
    on one handle and all scales in one list, against the fp64 Gram oracle."""
    gen = torch.Generator().manual_seed(205)
    base = torch.randn((300, 520), generator=gen)
    scales = (1e-30, 1e-20, 1e-6, 1e-3, 1.0, 1e3, 1e15, 1e30)
    for scale in scales:
        x = (base * scale).cuda()
        o = torch.empty_like(x)
        handle.gram_newton_schulz([x], [o])
        assert handle.status()[0] == 0
        assert bool(torch.isfinite(o).all()), scale
        ref = og.gram_newton_schulz(x.cpu().numpy().astype(np.float64))
        assert rel_fro(o.cpu().numpy(), ref) <= NS_TOL, scale
    xs = [(base[:, : 300 + 20 * k] * sc).cuda() for k, sc in enumerate(scales)]
    outs = [torch.empty_like(x) for x in xs]
    handle.gram_newton_schulz(xs, outs)
    assert handle.status()[0] == 0
    for x, o, sc in zip(xs, outs, scales):
        assert rel_fro(o.cpu().numpy(), og.gram_newton_schulz(x.cpu().numpy().astype(np.float64))) <= NS_TOL, sc


@pytest.mark.parametrize("kw", [dict(), dict(nesterov=False), dict(wd=0.1), dict(scale_mode=2),
                                dict(ns_steps=3, restarts=(1,))])
def test_gram_step(handle, kw):
    shapes = [(384, 1000), (1000, 384), (520, 520), (64, 1500)]
    Ws, Gs, Ms = _inputs(shapes, 207)
    Wd, Gd, Md = _dev(Ws), _dev(Gs), _dev(Ms)
    kw = dict(kw)
    ns = kw.pop("ns_steps", 5)
    rs = kw.pop("restarts", None)
    wd = kw.pop("wd", 0.0)
    handle.step(Wd, Gd, Md, lr=0.05, mu=0.9, ns_steps=ns, weight_decay=wd, backend="gram", restarts=rs, **kw)
    rc, flags = handle.status(len(shapes))
    assert rc == 0 and not any(flags)
    for i, s in enumerate(shapes):
        ref = og.muon_step_gram(Ws[i].numpy(), Gs[i].numpy(), Ms[i].numpy(), lr=F32(0.05), mu=F32(0.9),
                                wd=F32(wd), ns_steps=ns, restarts=(2,) if rs is None else rs, **kw)
        W0 = Ws[i].numpy().astype(np.float64)
        assert_momentum(Md[i].cpu().numpy(), ref["M"])
        e = rel_fro(Wd[i].cpu().numpy().astype(np.float64) - W0, ref["W"] - W0)
        assert e <= NS_TOL, (s, kw, e)


def test_gram_and_direct_backends_agree(handle):
    """Same step with both backends on one handle (the plan switches) and
    the same coefficient table (the Gram backend's default, Polar Express):
    both meet the bar and agree with each other."""
    shapes = [(512, 1536), (1536, 512)]
    Ws, Gs, Ms = _inputs(shapes, 209)
    table = dm.dmuon_polar_express_coefficients(5)
    res = {}
    for backend in ("direct", "gram", "direct"):
        Wd, Gd, Md = _dev(Ws), _dev(Gs), _dev(Ms)
        handle.step(Wd, Gd, Md, backend=backend, coeffs=table)
        assert handle.status()[0] == 0
        res.setdefault(backend, []).append([w.cpu() for w in Wd])
    for a, b in zip(res["direct"][0], res["direct"][1]):
        assert torch.equal(a, b)   # switching the plan back gives the same bits
    for a, b, w0 in zip(res["gram"][0], res["direct"][0], Ws):
        assert rel_fro((a - w0).numpy(), (b - w0).numpy()) <= 2 * NS_TOL


@pytest.mark.parametrize("shapes,launches", [
    # 4 (momentum pass, norm, redo pass, its norm) + window [0, 2) (X X^T, Z W R', Z Q') + Q X
    # + window [2, 4) (the same) + Q X + window [4, 5) (X X^T, Z) + final Q X, whatever the aspect ratio
    ([(300, 900), (700, 300)], 21),
    ([(300, 500), (700, 400)], 21),
])
def test_gram_deterministic_and_launch_count(handle, shapes, launches):
    Ws, Gs, Ms = _inputs(shapes, 211)
    Gd = _dev(Gs)
    outs = []
    for _ in range(2):
        Wd, Md = _dev(Ws), _dev(Ms)
        before = dm.dmuon_launch_count(handle.h)
        handle.step(Wd, Gd, Md, backend="gram")
        torch.cuda.synchronize()
        assert dm.dmuon_launch_count(handle.h) - before == launches
        outs.append([t.cpu() for t in Wd + Md])
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    assert handle.status()[0] == 0


def _spiked(shape, seed):
    """Gaussian bulk plus a rank-16 spike with singular values log-spaced
    from 1e2 down to 1e-3 (the spiked workload's construction)."""
    rng = np.random.default_rng(seed)
    r, c = shape
    Uq, _ = np.linalg.qr(rng.standard_normal((r, 16)))
    Vq, _ = np.linalg.qr(rng.standard_normal((c, 16)))
    G = rng.standard_normal((r, c)) + (Uq * np.logspace(2, -3, 16)) @ Vq.T
    return torch.from_numpy(np.ascontiguousarray(G, dtype=np.float32))


@pytest.mark.parametrize("path", ["gram", "gram_no_restart", "direct", "small"])
def test_polar_express_table(path):
    """The library's Polar Express table (dmuon_polar_express_coefficients)
    on the GPU paths against the fp64 oracles run with the oracle's own table
    (oracle.polar_express, an independent construction): the Gram backend with
    its default restart and with none, the direct iteration, the small-matrix
    kernel; random and spiked inputs (a square one included), ragged shapes."""
    from oracle import polar_express as pe
    table = dm.dmuon_polar_express_coefficients(5)
    ref_table = pe.polar_express_rows(5)
    assert dm.dmuon_gram_check_coefficients(5, table)[0]
    if path == "small":
        shapes, spiked = [(64, 256), (128, 512), (300, 100), (37, 5)], [(128, 512), (100, 100)]
    else:
        shapes = [(300, 700), (700, 300), (513, 1000), (200, 200), (255, 2050), (1024, 4096)]
        spiked = [(300, 1000), (1000, 300), (512, 512)]
    gen = torch.Generator().manual_seed(211)
    ins = [torch.randn(s, generator=gen) for s in shapes] + [_spiked(s, 212 + i) for i, s in enumerate(spiked)]
    shapes = shapes + spiked
    outs = [torch.empty(s, device="cuda") for s in shapes]
    with dm.Handle(0) as h2:
        if path != "small":
            dm.dmuon_set_small_path(h2.h, False)
        if path.startswith("gram"):
            restarts = () if path == "gram_no_restart" else None
            h2.gram_newton_schulz(_dev(ins), outs, ns_steps=5, coeffs=table, restarts=restarts)
        else:
            h2.newton_schulz(_dev(ins), outs, ns_steps=5, coeffs=table)
        assert h2.status()[0] == 0
        if path == "small":
            assert "small-matrix kernel %d;" % len(shapes) in dm.dmuon_plan_summary(h2.h)
    for x, o, s in zip(ins, outs, shapes):
        if path.startswith("gram"):
            restarts = () if path == "gram_no_restart" else (2,)
            ref = og.gram_newton_schulz(x.numpy(), 5, coeffs=ref_table, restarts=restarts)
        else:
            ref = oracle.newton_schulz(x.numpy(), 5, coeffs=ref_table)
        e = rel_fro(o.cpu().numpy(), ref)
        assert e <= NS_TOL, (path, s, e)


GRAM_STRESS = ["ill_300x700_r164", "ill_128x4096_r1e3", "ill_500x500_r1e4", "gauss_200x200", "gauss_384x384",
               "spiked_512x512", "spiked_700x300"]


def _stress_input(name):
    """The inputs on which the fp16 Gram form is weakest: singular values
    spread log-uniformly over [1/ratio, 1] (ratio 164 is the spread
    1.1e-3 ... 0.18 of a normalised 300 x 700 matrix), square Gaussian
    matrices (singular values down to ~0) and Gaussian bulks with a rank-16
    spike from 1e2 down to 1e-3."""
    from _parity import spectrum_matrix
    kind, shape = name.split("_")[:2]
    r, c = (int(v) for v in shape.split("x"))
    if kind == "ill":
        ratio = float(name.split("_r")[1])
        return torch.from_numpy(spectrum_matrix(r, c, ratio, 41))
    if kind == "gauss":
        return torch.randn((r, c), generator=torch.Generator().manual_seed(43))
    return _spiked((r, c), 45)


@pytest.mark.parametrize("restarts", [(2,), (), (1,)])
@pytest.mark.parametrize("table", ["polar_express", "you"])
def test_gram_stress_inputs(handle, table, restarts):
    """Every stress input, both tables, the default restart and none (both
    run as windows of 2 + 2 + 1 steps) and a restart before the second step
    (windows of 1 + 2 + 2): each within 3e-2 of the fp64 Gram oracle."""
    from oracle import polar_express as pe
    coeffs = None if table == "polar_express" else oracle.coefficient_rows(5)
    ins = [_stress_input(n) for n in GRAM_STRESS]
    outs = [torch.empty_like(x, device="cuda") for x in ins]
    handle.gram_newton_schulz(_dev(ins), outs, ns_steps=5, coeffs=coeffs, restarts=restarts)
    assert handle.status()[0] == 0
    ref_coeffs = pe.polar_express_rows(5) if coeffs is None else coeffs
    for name, x, o in zip(GRAM_STRESS, ins, outs):
        ref = og.gram_newton_schulz(x.numpy().astype(np.float64), 5, coeffs=ref_coeffs, restarts=restarts)
        e = rel_fro(o.cpu().numpy(), ref)
        assert e <= NS_TOL, (name, table, restarts, e)


def test_gram_argument_errors(handle):
    x = torch.randn((300, 900), device="cuda")
    o = torch.empty_like(x)
    p = [x.data_ptr()], [o.data_ptr()], [(300, 900)]
    before = dm.dmuon_launch_count(handle.h)
    # a window of 8 steps without restart: gain prod |a| ~ 1.1e4 > 8192
    assert dm.dmuon_gram_newton_schulz_ptrs(handle.h, *p, ns_steps=1, coeffs=[(1.0, 25.0, 0.0)],
                                            check=False) == -1
    assert "fp16" in dm.dmuon_last_error(handle.h)   # x + 25 x^3: singular values past kappa R's range
    assert dm.dmuon_gram_newton_schulz_ptrs(handle.h, *p, ns_steps=1, coeffs=[(0.0, 0.0, 1.0)], check=False) == -1
    assert "1/64" in dm.dmuon_last_error(handle.h)
    assert dm.dmuon_launch_count(handle.h) == before
    # eight steps without a restart run as four windows of two steps, the same function
    for restarts in ((), (3, 6)):
        assert dm.dmuon_gram_newton_schulz_ptrs(handle.h, *p, ns_steps=8, restarts=restarts, check=False) == 0
        assert handle.status()[0] == 0
        ref = og.gram_newton_schulz(x.cpu().numpy(), 8, restarts=restarts)
        assert rel_fro(o.cpu().numpy(), ref) <= NS_TOL


def test_gram_step_in_cuda_graph(handle):
    shapes = [(384, 1000), (600, 300)]
    Ws, Gs, Ms = _inputs(shapes, 213)
    Wa, Ga, Ma = _dev(Ws), _dev(Gs), _dev(Ms)
    for _ in range(3):
        handle.step(Wa, Ga, Ma, backend="gram")
    torch.cuda.synchronize()
    with dm.Handle(0) as h2:
        Wb, Gb, Mb = _dev(Ws), _dev(Gs), _dev(Ms)
        h2.step(Wb, Gb, Mb, backend="gram")
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            h2.step(Wb, Gb, Mb, backend="gram")
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        assert h2.status()[0] == 0
        for a, b in zip(Wa + Ma, Wb + Mb):
            assert torch.equal(a, b)


@pytest.mark.slow
def test_gram_full_llama3_8b_sampled(handle):
    """All 224 Llama-3-8B matrices with the Gram backend (bench launch
    configuration); sampled matrices against the Gram oracle."""
    w = workloads.get("llama3_8b")
    n = len(w.shapes)
    dev = "cuda"
    Wd = [workloads.weight(w, i, dev) for i in range(n)]
    Md = [workloads.momentum(w, i, dev) for i in range(n)]
    Gd = [workloads.grad(w, i, 0, dev) for i in range(n)]
    sample = [0, 1, 4, 6, 218]
    W0 = {i: Wd[i].cpu() for i in sample}
    M0 = {i: Md[i].cpu() for i in sample}
    with dm.Handle(0) as h2:
        h2.step(Wd, Gd, Md, backend="gram")
        assert h2.status()[0] == 0
    for i in sample:
        ref = og.muon_step_gram(W0[i].numpy(), Gd[i].cpu().numpy(), M0[i].numpy(), lr=F32(0.02), mu=F32(0.95))
        w0 = W0[i].numpy().astype(np.float64)
        assert_momentum(Md[i].cpu().numpy(), ref["M"])
        e = rel_fro(Wd[i].cpu().numpy().astype(np.float64) - w0, ref["W"] - w0)
        assert e <= NS_TOL, (i, w.shapes[i], e)
    del Wd, Md, Gd
    torch.cuda.empty_cache()


def test_gram_nonfinite_flags_in_caller_order(handle):
    shapes = [(300, 500), (700, 300), (260, 900)]
    Ws = [torch.zeros(s, device="cuda") for s in shapes]
    Gs = [torch.randn(s, device="cuda") for s in shapes]
    Ms = [torch.zeros(s, device="cuda") for s in shapes]
    Gs[1][5, 7] = float("nan")
    handle.step(Ws, Gs, Ms, backend="gram")
    rc, flags = handle.status(3)
    assert rc == -5 and flags == [0, 1, 0]
    assert handle.status(3) == (0, [0, 0, 0])


def test_gram_wait_timeout_is_reported_and_context_recovers(handle):
    """A 1 ns wait limit makes the Gram-space (and Apply) kernels give up at
    their first non-immediate wait, drain their own copies and MMAs, free
    TMEM and return; the host reads DMUON_ERR_TIMEOUT, and with the default
    limit restored the next step meets the bar again."""
    shapes = [(384, 1000), (600, 300)]
    Ws, Gs, Ms = _inputs(shapes, 215)
    dm.dmuon_set_wait_timeout(handle.h, 1)
    try:
        handle.step(_dev(Ws), _dev(Gs), _dev(Ms), backend="gram")
        rc, _ = handle.status(2)
    finally:
        dm.dmuon_set_wait_timeout(handle.h, 0)
    assert rc == -6
    assert handle.status(2)[0] == 0
    Wd, Gd, Md = _dev(Ws), _dev(Gs), _dev(Ms)
    handle.step(Wd, Gd, Md, backend="gram")
    assert handle.status(2)[0] == 0
    for i in range(2):
        ref = og.muon_step_gram(Ws[i].numpy(), Gs[i].numpy(), Ms[i].numpy(), lr=F32(0.02), mu=F32(0.95))
        W0 = Ws[i].numpy().astype(np.float64)
        assert rel_fro(Wd[i].cpu().numpy().astype(np.float64) - W0, ref["W"] - W0) <= NS_TOL


def _gram_full_size_sampled(name, sample):
    w = workloads.get(name)
    n = len(w.shapes)
    dev = "cuda"
    Wd = [workloads.weight(w, i, dev) for i in range(n)]
    Md = [workloads.momentum(w, i, dev) for i in range(n)]
    with dm.Handle(0) as h2:
        for step in range(w.warm_steps):
            Gw = [workloads.grad(w, i, step, dev) for i in range(n)]
            h2.step(Wd, Gw, Md, backend="gram")
            del Gw
        Gd = [workloads.grad(w, i, w.warm_steps, dev) for i in range(n)]
        W0 = {i: Wd[i].cpu() for i in sample}
        M0 = {i: Md[i].cpu() for i in sample}
        h2.step(Wd, Gd, Md, backend="gram")
        assert h2.status()[0] == 0
    for i in sample:
        ref = og.muon_step_gram(W0[i].numpy(), Gd[i].cpu().numpy(), M0[i].numpy(), lr=F32(0.02), mu=F32(0.95))
        w0 = W0[i].numpy().astype(np.float64)
        assert_momentum(Md[i].cpu().numpy(), ref["M"])
        e = rel_fro(Wd[i].cpu().numpy().astype(np.float64) - w0, ref["W"] - w0)
        assert e <= NS_TOL, (name, i, w.shapes[i], e)
    del Wd, Md, Gd
    torch.cuda.empty_cache()


@pytest.mark.slow
def test_gram_full_spiked_4096_sampled(handle):
    """Singular values spread over 1e-3..1e2 (rank-16 spike): the widest
    spectrum of the workloads, through the fp16 Gram window."""
    _gram_full_size_sampled("spiked_4096", [0, 63])


@pytest.mark.slow
def test_gram_full_tp_70b_mixed_sampled(handle):
    """The 28672x8192 matrix (m = 8192, the largest Gram window) and packed
    64x256 matrices (small-matrix kernel) in one call."""
    _gram_full_size_sampled("tp_70b_mixed", [0, 1, 300, 512])


def test_gram_chunking_is_bitwise_neutral(handle):
    """One chunk, many chunks, and many chunks with the next chunk's
    momentum pass overlapped (chunks alternating between two workspaces that
    hold their Gram-window buffers) give the same bits."""
    gen = torch.Generator().manual_seed(217)
    shapes = [(300, 500), (500, 300), (257, 257), (200, 900), (900, 200), (130, 900)]
    Ws = [torch.rand(s, generator=gen) - 0.5 for s in shapes]
    Gs = [torch.randn(s, generator=gen) for s in shapes]
    Ms = [torch.randn(s, generator=gen) for s in shapes]
    res = {}
    for elems, overlap in ((1 << 29, False), (200_000, True), (200_001, False)):
        with dm.Handle(0) as h2:
            dm.dmuon_set_chunk_elements(h2.h, elems)
            dm.dmuon_set_overlap(h2.h, overlap)
            Wd, Gd, Md = _dev(Ws), _dev(Gs), _dev(Ms)
            h2.step(Wd, Gd, Md, backend="gram")
            assert h2.status()[0] == 0
            summary = dm.dmuon_plan_summary(h2.h)
            res[elems] = ([x.cpu() for x in Wd + Md], summary)
    import re
    n_chunks = {k: int(re.search(r"chunks (\d+) ", v[1]).group(1)) for k, v in res.items()}
    assert n_chunks[1 << 29] == 1 and n_chunks[200_000] > 2
    for key in (200_000, 200_001):
        for a, b in zip(res[1 << 29][0], res[key][0]):
            assert torch.equal(a, b)

"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Same seeded inputs on both sides.  Bars (per matrix):
  momentum buffer   relative Frobenius error <= 1e-6   (fp32 arithmetic)
  NS output O and the weight update W' - W
                    relative Frobenius error <= 3e-2   (bf16 tensor cores)
The small cases span several 128x256 tiles and ragged tails; the full-size
cases run every matrix of a workload in the bench's launch configuration
and compare sampled matrices with the oracle.
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
F32 = lambda x: float(np.float32(x))  # noqa: E731  (the ABI takes fp32 scalars)


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


def _to_dev(ts):
    return [t.clone().cuda() for t in ts]


def _step_and_check(handle, Ws, Gs, Ms, lr=0.02, mu=0.95, ns_steps=5, wd=0.0, nesterov=True,
                    scale_mode=0, coeffs=None, ns_tol=NS_TOL):
    Wd, Gd, Md = _to_dev(Ws), _to_dev(Gs), _to_dev(Ms)
    handle.step(Wd, Gd, Md, lr=lr, mu=mu, ns_steps=ns_steps, weight_decay=wd,
                nesterov=nesterov, scale_mode=scale_mode, coeffs=coeffs)
    rc, flags = handle.status(len(Ws))
    assert rc == 0 and not any(flags)
    worst = 0.0
    for i in range(len(Ws)):
        ref = oracle.muon_step(Ws[i].numpy(), Gs[i].numpy(), Ms[i].numpy(), lr=F32(lr), mu=F32(mu),
                               wd=F32(wd), ns_steps=ns_steps, coeffs=coeffs, nesterov=nesterov,
                               scale_mode=scale_mode)
        W0 = Ws[i].numpy().astype(np.float64)
        assert_momentum(Md[i].cpu().numpy(), ref["M"], "matrix %d" % i)
        e_upd = rel_fro(Wd[i].cpu().numpy().astype(np.float64) - W0, ref["W"] - W0)
        e_w = rel_fro(Wd[i].cpu().numpy(), ref["W"])
        assert e_upd <= ns_tol, ("update", i, Ws[i].shape, e_upd)
        assert e_w <= ns_tol, ("weight", i, e_w)
        worst = max(worst, e_upd)
    return worst


def test_tinymlp_d128_step(handle):
    w = workloads.get("tinymlp_d128")
    n = len(w.shapes)
    Ws = [workloads.weight(w, i) for i in range(n)]
    Gs = [workloads.grad(w, i) for i in range(n)]
    Ms = [workloads.momentum(w, i) for i in range(n)]
    worst = _step_and_check(handle, Ws, Gs, Ms)
    assert worst < NS_TOL


def test_tinymlp_d512_three_steps(handle):
    """Zero momentum, three steps with fresh gradients; the oracle runs the
    same three steps from the same initial state."""
    w = workloads.get("tinymlp_d512")
    n = len(w.shapes)
    W0 = [workloads.weight(w, i) for i in range(n)]
    M0 = [workloads.momentum(w, i) for i in range(n)]
    Wd, Md = _to_dev(W0), _to_dev(M0)
    Wr = [x.numpy().astype(np.float64) for x in W0]
    Mr = [x.numpy().astype(np.float64) for x in M0]
    for step in range(w.warm_steps + 1):
        Gs = [workloads.grad(w, i, step) for i in range(n)]
        Gd = _to_dev(Gs)
        handle.step(Wd, Gd, Md, lr=0.02, mu=0.95, ns_steps=5)
        for i in range(n):
            out = oracle.muon_step(Wr[i], Gs[i].numpy(), Mr[i], lr=F32(0.02), mu=F32(0.95))
            # the momentum state between steps is an fp32 buffer, on both sides
            Wr[i], Mr[i] = out["W"], out["M"].astype(np.float32)
    rc, _ = handle.status()
    assert rc == 0
    for i in range(n):
        W0i = W0[i].numpy().astype(np.float64)
        assert_momentum(Md[i].cpu().numpy(), Mr[i])
        assert rel_fro(Wd[i].cpu().numpy().astype(np.float64) - W0i, Wr[i] - W0i) <= NS_TOL


RAGGED = [(1, 1), (1, 37), (37, 1), (3, 5), (5, 3), (64, 256), (256, 64), (128, 512),
          (129, 257), (300, 700), (700, 300), (200, 200), (513, 1000), (1000, 513),
          (255, 2050), (8, 4100), (384, 384), (640, 96)]


def test_newton_schulz_ragged_shapes(handle):
    gen = torch.Generator().manual_seed(7)
    ins = [torch.randn(s, generator=gen) for s in RAGGED]
    outs = [torch.empty(s, device="cuda") for s in RAGGED]
    handle.newton_schulz(_to_dev(ins), outs)
    rc, _ = handle.status()
    assert rc == 0
    for x, o, s in zip(ins, outs, RAGGED):
        ref = oracle.newton_schulz(x.numpy())
        e = rel_fro(o.cpu().numpy(), ref)
        assert e <= NS_TOL, (s, e)


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_tile_modes_match_oracle(handle, mode):
    """Single-CTA 128x256 tiles (mode 1), CTA-pair 256x256 tiles (mode 2) and
    single-CTA 128x128 tiles (mode 3) all meet the bar on ragged shapes and a
    full step (the small-matrix kernel off, so that the small shapes run
    through these tiles too)."""
    gen = torch.Generator().manual_seed(23)
    ins = [torch.randn(s, generator=gen) for s in RAGGED]
    outs = [torch.empty(s, device="cuda") for s in RAGGED]
    with dm.Handle(0) as h2:
        dm.dmuon_set_tile_mode(h2.h, mode)
        dm.dmuon_set_small_path(h2.h, False)
        h2.newton_schulz(_to_dev(ins), outs)
        assert h2.status()[0] == 0
        assert (("pairs" in dm.dmuon_plan_summary(h2.h)) == (mode == 2))
        assert (("128x128" in dm.dmuon_plan_summary(h2.h)) == (mode == 3))
        for x, o, s in zip(ins, outs, RAGGED):
            e = rel_fro(o.cpu().numpy(), oracle.newton_schulz(x.numpy()))
            assert e <= NS_TOL, (mode, s, e)
        shapes = [(512, 128), (128, 512), (300, 1000), (1000, 300)]
        Ws = [torch.rand(s, generator=gen) - 0.5 for s in shapes]
        Gs = [torch.randn(s, generator=gen) for s in shapes]
        Ms = [torch.randn(s, generator=gen) for s in shapes]
        _step_and_check(h2, Ws, Gs, Ms)


@pytest.mark.parametrize("mode", [1, 3])
@pytest.mark.parametrize("seed", [61, 62])
def test_single_cta_tiles_random_lists(mode, seed):
    """Seeded random lists (short sides 1-700 on both sides of every 128 and
    256 boundary, long sides up to 1500, both orientations) with 1-7 steps
    and the fused and per-phase launches, on 128x256 (mode 1) and 128x128
    (mode 3) single-CTA tiles, against the fp64 oracle."""
    rng = np.random.default_rng(seed)
    shapes = []
    for _ in range(9):
        m = int(rng.choice([int(rng.integers(1, 700)), 128, 129, 255, 256, 257, 383, 384, 385]))
        n = int(rng.integers(m, 1500))
        shapes.append((m, n) if rng.random() < 0.5 else (n, m))
    gen = torch.Generator().manual_seed(seed)
    Ws = [torch.rand(sh, generator=gen) - 0.5 for sh in shapes]
    Gs = [torch.randn(sh, generator=gen) for sh in shapes]
    Ms = [torch.randn(sh, generator=gen) for sh in shapes]
    ns = int(rng.integers(1, 8))
    for fused in (True, False):
        with dm.Handle(0) as h2:
            dm.dmuon_set_tile_mode(h2.h, mode)
            dm.dmuon_set_small_path(h2.h, False)
            dm.dmuon_set_fused_phases(h2.h, fused)
            _step_and_check(h2, Ws, Gs, Ms, ns_steps=ns)
            assert ("128x128" in dm.dmuon_plan_summary(h2.h)) == (mode == 3)


# Rows isolating each term.  Every row keeps a >= 1/64 (the library refuses rows without the
# identity part, which the unscaled fp16 Z needs); with the inputs below -- rank two plus a little
# noise, normalised singular values ~0.83 and ~0.55 -- the b and c terms of the second and third
# rows carry 90 % and more of the output.  The last row mixes all three terms; its polynomial
# 0.5 s - 0.25 s^3 + 0.125 s^5 stays away from zero on (0, 1].
SINGLE_TERM_ROWS = [(1.0, 0.0, 0.0), (1.0 / 64, 1.0, 0.0), (1.0 / 64, 0.0, 1.0), (0.5, -0.25, 0.125)]
TERM_SHAPES = {
    "pair": [(1, 300), (300, 1), (64, 64), (130, 700), (700, 130), (257, 257), (520, 520)],
    "single": [(1, 300), (64, 64), (130, 700), (700, 130), (257, 257)],
    "narrow": [(1, 300), (64, 64), (130, 700), (700, 130), (257, 257), (300, 520)],
    "small": [(1, 300), (300, 1), (64, 64), (100, 500), (500, 100), (128, 128)],
    "gram": [(1, 300), (64, 64), (130, 700), (700, 130), (257, 257), (520, 1100)],
}


@pytest.mark.parametrize("path", ["pair", "single", "narrow", "small", "gram"])
@pytest.mark.parametrize("row", SINGLE_TERM_ROWS)
def test_each_term_of_the_step(path, row):
    """One Newton-Schulz step with one term of X' = aX + b(XX^T)X + c(XX^T)^2 X
    at a time, on every path (CTA-pair and single-CTA GEMM kernels, the
    small-matrix kernel, the Gram-space kernels), against the fp64 oracle:
    a dropped, doubled or mis-signed term in any epilogue fails here on its own.
    Shapes include one-row and one-column matrices, one 64-wide tile, and
    ragged tiles on both sides of the diagonal."""
    shapes = TERM_SHAPES[path]
    gen = torch.Generator().manual_seed(47)
    ins = []
    for r, c in shapes:   # rank two (weights 3 and 2) plus noise of norm ~0.05
        u, v = torch.randn((r, 2), generator=gen), torch.randn((c, 2), generator=gen)
        u, v = torch.linalg.qr(u)[0] if r > 1 else u / u.norm(), torch.linalg.qr(v)[0] if c > 1 else v / v.norm()
        low = 3.0 * torch.outer(u[:, 0], v[:, 0]) + (2.0 * torch.outer(u[:, 1], v[:, 1]) if min(r, c) > 1 else 0.0)
        ins.append((low + 0.05 * torch.randn((r, c), generator=gen) / (r * c) ** 0.5).contiguous())
    outs = [torch.empty(s, device="cuda") for s in shapes]
    with dm.Handle(0) as h2:
        if path == "pair":
            dm.dmuon_set_tile_mode(h2.h, 2)
        if path == "single":
            dm.dmuon_set_tile_mode(h2.h, 1)
        if path == "narrow":
            dm.dmuon_set_tile_mode(h2.h, 3)
        if path != "small":
            dm.dmuon_set_small_path(h2.h, False)
        if path == "gram":
            h2.gram_newton_schulz(_to_dev(ins), outs, ns_steps=1, coeffs=[row], restarts=[])
        else:
            h2.newton_schulz(_to_dev(ins), outs, ns_steps=1, coeffs=[row])
        rc, _ = h2.status()
        assert rc == 0
        if path == "small":
            assert "small-matrix kernel %d;" % len(shapes) in dm.dmuon_plan_summary(h2.h)
    for x, o, s in zip(ins, outs, shapes):
        ref = oracle.newton_schulz(x.numpy(), 1, coeffs=[row])
        e = rel_fro(o.cpu().numpy(), ref)
        assert e <= 1e-2, (path, row, s, e)


SCALES = (1e-30, 1e-20, 1e-6, 1e-3, 1.0, 1e3, 1e15, 1e30)


def test_newton_schulz_scaled_inputs(handle):
    """The normalisation is folded into the first products, with the fp16
    iterate prescaled by a power of two from max |U| (and the iterate after
    the first product rescaled when ||U|| is far below eps): inputs over the
    whole fp32 range (scales 1e-30 ... 1e30, one call per scale on the same
    handle, so the prescale kept from the previous call misses every time)
    meet the bar against the oracle, whose normaliser has no range limit;
    then all scales in one list."""
    gen = torch.Generator().manual_seed(9)
    base = torch.randn((300, 520), generator=gen)
    for scale in SCALES:
        x = (base * scale).cuda()
        o = torch.empty_like(x)
        handle.newton_schulz([x], [o])
        assert handle.status()[0] == 0
        assert bool(torch.isfinite(o).all()), scale
        assert rel_fro(o.cpu().numpy(), oracle.newton_schulz(x.cpu().numpy().astype(np.float64))) <= NS_TOL, scale
    xs = [(base[: 200 + 10 * k] * sc).cuda() for k, sc in enumerate(SCALES)]
    os_ = [torch.empty_like(x) for x in xs]
    handle.newton_schulz(xs, os_)
    assert handle.status()[0] == 0
    for x, o, sc in zip(xs, os_, SCALES):
        assert rel_fro(o.cpu().numpy(), oracle.newton_schulz(x.cpu().numpy().astype(np.float64))) <= NS_TOL, sc


def test_step_scaled_inputs_and_prescale_redo(handle):
    """Muon steps whose gradients jump by many orders of magnitude from one
    step to the next on the same handle: the prescale kept from the previous
    step misses, the redo pass rewrites X0, and every step meets the bar
    (momentum element by element)."""
    gen = torch.Generator().manual_seed(19)
    shapes = [(384, 640), (640, 384)]
    Ws = [torch.rand(s, generator=gen) - 0.5 for s in shapes]
    Gb = [torch.randn(s, generator=gen) for s in shapes]
    Wd, Md = _to_dev(Ws), [torch.zeros(s, device="cuda") for s in shapes]
    for scale in (1.0, 1e-25, 1e20, 1e-3, 1e-3):
        Gs = [g * scale for g in Gb]
        W0 = [w.cpu() for w in Wd]
        M0 = [m.cpu() for m in Md]
        handle.step(Wd, _to_dev(Gs), Md)
        assert handle.status()[0] == 0
        for i in range(2):
            ref = oracle.muon_step(W0[i].numpy(), Gs[i].numpy(), M0[i].numpy(), lr=F32(0.02), mu=F32(0.95))
            assert_momentum(Md[i].cpu().numpy(), ref["M"], "scale %g matrix %d" % (scale, i))
            w0 = W0[i].numpy().astype(np.float64)
            e = rel_fro(Wd[i].cpu().numpy().astype(np.float64) - w0, ref["W"] - w0)
            assert e <= NS_TOL, (scale, i, e)


@pytest.mark.parametrize("f16_iters", [3, 64])
@pytest.mark.parametrize("ratio", [1e2, 1e3, 1e4])
@pytest.mark.parametrize("table", ["you", "polar_express"])
def test_ill_conditioned_inputs(handle, ratio, table, f16_iters):
    """Inputs whose singular values spread log-uniformly over [1/ratio, 1]
    (wide, tall and square; ratio up to 1e4), with the printed table and the
    Polar Express table, fp16 operands in the first three iterations (the
    default) or in all: the output stays within the bar."""
    from _parity import spectrum_matrix
    from oracle import polar_express as pe
    coeffs = None if table == "you" else dm.dmuon_polar_express_coefficients(5)
    ref_coeffs = None if table == "you" else pe.polar_express_rows(5)
    shapes = [(300, 700), (700, 300), (500, 500), (128, 4096)]
    ins = [torch.from_numpy(spectrum_matrix(r, c, ratio, 31 + k)) for k, (r, c) in enumerate(shapes)]
    outs = [torch.empty(s, device="cuda") for s in shapes]
    dm.dmuon_set_fp16_iterations(handle.h, f16_iters)
    try:
        handle.newton_schulz([x.cuda() for x in ins], outs, coeffs=coeffs)
    finally:
        dm.dmuon_set_fp16_iterations(handle.h, 3)
    assert handle.status()[0] == 0
    for x, o, s in zip(ins, outs, shapes):
        ref = oracle.newton_schulz(x.numpy().astype(np.float64), 5, coeffs=ref_coeffs)
        e = rel_fro(o.cpu().numpy(), ref)
        assert e <= NS_TOL, (s, ratio, table, e)


def test_fp16_iterations_knob(handle):
    """Each iteration's operand format follows the knob: on a Gaussian
    input, fp16 everywhere is the most accurate and fp16 in the first
    iteration only the least, all within the bar; fused and per-phase
    launches agree bitwise at every setting; 0 is refused."""
    x = torch.randn((512, 1536), generator=torch.Generator().manual_seed(71))
    ref = oracle.newton_schulz(x.numpy().astype(np.float64))
    errs = {}
    for iters in (1, 3, 64):
        outs = []
        for fused in (1, 0):
            o = torch.empty((512, 1536), device="cuda")
            dm.dmuon_set_fp16_iterations(handle.h, iters)
            dm.dmuon_set_fused_phases(handle.h, fused)
            try:
                handle.newton_schulz([x.cuda()], [o])
            finally:
                dm.dmuon_set_fp16_iterations(handle.h, 3)
                dm.dmuon_set_fused_phases(handle.h, 2)
            assert handle.status()[0] == 0
            outs.append(o.cpu())
        assert torch.equal(outs[0], outs[1])
        errs[iters] = rel_fro(outs[0].numpy(), ref)
    assert errs[64] < errs[3] < errs[1] <= NS_TOL, errs
    with pytest.raises(dm.DmuonError):
        dm.dmuon_set_fp16_iterations(handle.h, 0)


def test_coefficient_table_outside_fp16_range_is_refused(handle):
    """A table whose iterate could leave fp16's range (x + 25 x^3 sends
    singular value 1 to 26, and kappa X X^T past 32768 on the next step) is
    refused on the host with the reason, before anything is launched."""
    x = torch.randn((200, 300), device="cuda")
    o = torch.zeros_like(x)
    before = dm.dmuon_launch_count(handle.h)
    rc = dm.dmuon_newton_schulz_ptrs(handle.h, [x.data_ptr()], [o.data_ptr()], [(200, 300)], ns_steps=3,
                                     coeffs=[(1.0, 25.0, 0.0)] * 3, check=False)
    assert rc == -1 and "fp16" in dm.dmuon_last_error(handle.h)
    assert dm.dmuon_launch_count(handle.h) == before and float(o.abs().max()) == 0.0


def test_zero_input_gives_zero_output(handle):
    x = torch.zeros((260, 300), device="cuda")
    o = torch.full_like(x, 5.0)
    handle.newton_schulz([x], [o])
    assert float(o.abs().max()) == 0.0


@pytest.mark.parametrize("kw", [
    dict(ns_steps=0), dict(ns_steps=1), dict(ns_steps=2), dict(ns_steps=7),
    dict(nesterov=False), dict(wd=0.1), dict(scale_mode=1), dict(scale_mode=2),
    dict(coeffs=[(3.4445, -4.7750, 2.0315)] * 5),
    dict(ns_steps=3, coeffs=[(3.0, -3.2, 1.2), (2.5, -2.0, 0.5), (1.875, -1.25, 0.375)]),
])
def test_step_options(handle, kw):
    gen = torch.Generator().manual_seed(11)
    shapes = [(384, 200), (200, 640), (96, 96), (130, 70)]
    Ws = [torch.rand(s, generator=gen) - 0.5 for s in shapes]
    Gs = [torch.randn(s, generator=gen) for s in shapes]
    Ms = [torch.randn(s, generator=gen) for s in shapes]
    _step_and_check(handle, Ws, Gs, Ms, lr=0.05, mu=0.9, **kw)


def test_deterministic_bitwise(handle):
    w = workloads.get("tinymlp_d128")
    n = len(w.shapes)
    Ws = [workloads.weight(w, i) for i in range(n)]
    Gs = _to_dev([workloads.grad(w, i) for i in range(n)])
    Ms = [workloads.momentum(w, i) for i in range(n)]
    res = []
    for _ in range(2):
        Wd, Md = _to_dev(Ws), _to_dev(Ms)
        handle.step(Wd, Gs, Md)
        torch.cuda.synchronize()
        res.append(([x.cpu() for x in Wd], [x.cpu() for x in Md]))
    for a, b in zip(res[0][0] + res[0][1], res[1][0] + res[1][1]):
        assert torch.equal(a, b)


def test_chunking_is_bitwise_neutral(handle):
    """The same list stepped as one chunk and as many small chunks, with the
    next chunk's momentum pass overlapped or not, gives bitwise identical
    weights and momenta (each matrix's arithmetic does not depend on its
    neighbours); each chunk issues its own launches: momentum pass, norm,
    prescale redo pass, its norm, then one fused launch of all products."""
    gen = torch.Generator().manual_seed(29)
    shapes = [(300, 500), (500, 300), (257, 257), (64, 640), (640, 64), (130, 900)]
    Ws = [torch.rand(s, generator=gen) - 0.5 for s in shapes]
    Gs = [torch.randn(s, generator=gen) for s in shapes]
    Ms = [torch.randn(s, generator=gen) for s in shapes]
    res = {}
    for elems, overlap in ((1 << 29, True), (160_000, True), (160_001, False)):
        with dm.Handle(0) as h2:
            dm.dmuon_set_chunk_elements(h2.h, elems)
            dm.dmuon_set_overlap(h2.h, overlap)
            Wd, Gd, Md = _to_dev(Ws), _to_dev(Gs), _to_dev(Ms)
            before = dm.dmuon_launch_count(h2.h)
            h2.step(Wd, Gd, Md)
            assert h2.status()[0] == 0
            launches = dm.dmuon_launch_count(h2.h) - before
            summary = dm.dmuon_plan_summary(h2.h)
            res[elems] = ([x.cpu() for x in Wd], [x.cpu() for x in Md], launches, summary)
    assert res[1 << 29][2] == 5 and "chunks 1 " in res[1 << 29][3]   # a small list: fused automatically
    assert res[160_000][2] > 5 and res[160_000][2] % 5 == 0
    for key in (160_000, 160_001):   # overlapped and serial chunk schedules
        for a, b in zip(res[1 << 29][0] + res[1 << 29][1], res[key][0] + res[key][1]):
            assert torch.equal(a, b)


def _balance(summary):
    tail = summary.split("balance ")[1].split(";")[0].split()
    return {tail[i]: float(tail[i + 1]) for i in range(0, len(tail), 2)}


def test_items_dealt_evenly_for_one_llama_layer():
    """One Llama-3-8B layer per call: the Gram items (K = 4096 for q/k/v/o,
    K = 14336 for gate/up/down) are dealt longest-first to the least-loaded
    CTA pair, so the busiest pair's items cost at most 2 % more than the mean
    (a strided dealing of the same list gives ~10 %); the step still matches
    the oracle on a sampled matrix."""
    layer = [(4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096), (14336, 4096), (14336, 4096),
             (4096, 14336)]
    gen = torch.Generator(device="cuda").manual_seed(41)
    Ws = [torch.rand(s, generator=gen, device="cuda") - 0.5 for s in layer]
    Gs = [torch.randn(s, generator=gen, device="cuda") * 1e-3 for s in layer]
    Ms = [torch.randn(s, generator=gen, device="cuda") * 1e-3 for s in layer]
    W1, G1, M1 = Ws[1].cpu(), Gs[1].cpu(), Ms[1].cpu()
    with dm.Handle(0) as h2:
        h2.step(Ws, Gs, Ms)
        rc, flags = h2.status(len(layer))
        assert rc == 0 and not any(flags)
        summary = dm.dmuon_plan_summary(h2.h)
    bal = _balance(summary)
    assert "chunks 1 " in summary
    assert bal["gram"] <= 1.02, summary
    assert bal["gram2"] <= 1.05 and bal["apply"] <= 1.02, summary
    ref = oracle.muon_step(W1.numpy(), G1.numpy(), M1.numpy(), lr=F32(0.02), mu=F32(0.95))
    assert_momentum(Ms[1].cpu().numpy(), ref["M"])
    assert rel_fro(Ws[1].cpu().numpy() - W1.numpy(), ref["W"] - W1.numpy()) <= NS_TOL


@pytest.mark.parametrize("backend,tiles", [("direct", 2), ("direct", 1), ("direct", 3), ("gram", 2)])
def test_dealing_is_bitwise_neutral(backend, tiles):
    """Balanced and strided dealing of the same plan give bitwise equal
    weights and momenta (mixed K: tall, wide, square and ragged matrices in
    one chunk, more items than CTA pairs or CTAs in every phase), and the
    balanced plan is no less even than the strided one on this list (the
    busiest Gram processor: ~1.05 vs ~1.42 of the mean)."""
    gen = torch.Generator().manual_seed(43)
    shapes = [(6000, 2560), (2048, 2048), (768, 3000), (1536, 256), (640, 640), (300, 700), (1024, 130)]
    Ws = [torch.rand(s, generator=gen) - 0.5 for s in shapes]
    Gs = [torch.randn(s, generator=gen) for s in shapes]
    Ms = [torch.randn(s, generator=gen) for s in shapes]
    res = {}
    for balanced in (True, False):
        with dm.Handle(0) as h2:
            dm.dmuon_set_tile_mode(h2.h, tiles)
            dm.dmuon_set_balanced_dealing(h2.h, balanced)
            Wd, Gd, Md = _to_dev(Ws), _to_dev(Gs), _to_dev(Ms)
            h2.step(Wd, Gd, Md, backend=backend)
            assert h2.status()[0] == 0
            res[balanced] = ([x.cpu() for x in Wd], [x.cpu() for x in Md], _balance(dm.dmuon_plan_summary(h2.h)))
    for a, b in zip(res[True][0] + res[True][1], res[False][0] + res[False][1]):
        assert torch.equal(a, b)
    for phase in ("gram", "gram2", "apply"):
        assert res[True][2][phase] <= res[False][2][phase] + 1e-9, (res[True][2], res[False][2])


def test_step_recorded_in_cuda_graph(handle):
    """Three eager steps equal one eager step plus two replays of a graph
    that recorded the step, bitwise; capturing before the buffers were seen
    is refused with DMUON_ERR_ARG and records nothing."""
    w = workloads.get("tinymlp_d128")
    n = len(w.shapes)
    Ws = [workloads.weight(w, i) for i in range(n)]
    Gs = [workloads.grad(w, i) for i in range(n)]
    Ms = [workloads.momentum(w, i) for i in range(n)]
    Wa, Ga, Ma = _to_dev(Ws), _to_dev(Gs), _to_dev(Ms)
    for _ in range(3):
        handle.step(Wa, Ga, Ma)
    torch.cuda.synchronize()
    with dm.Handle(0) as h2:
        Wb, Gb, Mb = _to_dev(Ws), _to_dev(Gs), _to_dev(Ms)
        Wc, Gc, Mc = _to_dev(Ws), _to_dev(Gs), _to_dev(Ms)
        h2.step(Wb, Gb, Mb)            # plans and caches these buffers
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            h2.step(Wb, Gb, Mb)
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2):
            rc = dm.dmuon_step_ptrs(h2.h, [t.data_ptr() for t in Wc], [t.data_ptr() for t in Gc],
                                    [t.data_ptr() for t in Mc], [tuple(t.shape) for t in Wc],
                                    0.02, 0.95, 5, check=False)
        assert rc == -1 and "capture" in dm.dmuon_last_error(h2.h)
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        assert h2.status()[0] == 0
        for a, b in zip(Wa + Ma, Wb + Mb):
            assert torch.equal(a, b)
        for a, b in zip(Wc, Ws):
            assert torch.equal(a.cpu(), b)   # the refused capture changed nothing


def test_alternating_pointer_sets(handle):
    """Per-group calls (same shapes, different buffers) reuse cached pointer
    slots: 70 groups cycle through the 64 slots twice, so slots are evicted
    and refilled, and every group must still get its own result."""
    gen = torch.Generator().manual_seed(17)
    shapes = [(192, 320), (320, 96)]
    groups = []
    for _ in range(70):
        Ws = [torch.rand(s, generator=gen) - 0.5 for s in shapes]
        Gs = [torch.randn(s, generator=gen) for s in shapes]
        Ms = [torch.randn(s, generator=gen) for s in shapes]
        groups.append((Ws, Gs, Ms, _to_dev(Ws), _to_dev(Gs), _to_dev(Ms)))
    for _ in range(2):
        for Ws, Gs, Ms, Wd, Gd, Md in groups:
            handle.step(Wd, Gd, Md)
    assert handle.status()[0] == 0
    for Ws, Gs, Ms, Wd, Gd, Md in groups:
        W, M = [w.numpy() for w in Ws], [m.numpy() for m in Ms]
        for _ in range(2):
            for i in range(2):
                out = oracle.muon_step(W[i], Gs[i].numpy(), M[i], lr=F32(0.02), mu=F32(0.95))
                W[i], M[i] = out["W"], out["M"].astype(np.float32)  # fp32 state between steps
        for i in range(2):
            W0 = Ws[i].numpy().astype(np.float64)
            assert_momentum(Md[i].cpu().numpy(), M[i])
            assert rel_fro(Wd[i].cpu().numpy().astype(np.float64) - W0, W[i] - W0) <= NS_TOL


def test_nonfinite_is_flagged(handle):
    shapes = [(64, 96), (96, 64), (128, 128)]
    Ws = [torch.zeros(s, device="cuda") for s in shapes]
    Gs = [torch.ones(s, device="cuda") for s in shapes]
    Ms = [torch.zeros(s, device="cuda") for s in shapes]
    Gs[1][3, 5] = float("nan")
    handle.step(Ws, Gs, Ms)
    rc, flags = handle.status(3)
    assert rc == -5 and flags == [0, 1, 0]
    rc, flags = handle.status(3)  # flags are cleared by the read
    assert rc == 0 and flags == [0, 0, 0]


def test_argument_errors_with_live_handle(handle):
    h = handle.h
    W = torch.zeros((64, 64), device="cuda")
    G = torch.zeros((64, 64), device="cuda")
    M = torch.zeros((64, 64), device="cuda")
    p = lambda t: t.data_ptr()  # noqa: E731
    call = lambda **k: dm.dmuon_step_ptrs(h, k.get("w", [p(W)]), k.get("g", [p(G)]),  # noqa: E731
                                          k.get("m", [p(M)]), k.get("s", [(64, 64)]), 0.02, 0.95,
                                          k.get("ns", 5), scale_mode=k.get("sm", 0),
                                          coeffs=k.get("c"), check=False)
    before = dm.dmuon_launch_count(h)
    assert call(w=[p(W) + 4]) == -2
    assert call(s=[(0, 64)]) == -1
    assert call(s=[(40000, 40000)]) == -1          # short side above the limit
    assert call(s=[(64, (1 << 20) + 1)]) == -1     # long side above the limit
    assert call(ns=65) == -1
    assert call(ns=-1) == -1
    assert call(sm=3) == -1
    assert call(c=[(1.0, float("nan"), 0.0)] * 5) == -1
    assert call(g=[p(W)]) == -1
    assert call(w=[0]) == -1
    assert dm.dmuon_step_ptrs(h, [], [], [], [], 0.02, 0.95, check=False) == 0
    assert dm.dmuon_launch_count(h) == before  # nothing launched


@pytest.mark.parametrize("fused", [1, 0])
def test_wait_timeout_is_reported_and_context_recovers(handle, fused):
    """A 1 ns wait limit makes the GEMM kernels give up at their first
    non-immediate wait (an mbarrier, or in the fused launch a tile counter):
    they drain, free TMEM and return; the host reads DMUON_ERR_TIMEOUT, and
    with the default limit restored the next step is correct again.  Both
    the fused launch and the per-phase launches."""
    shapes = [(384, 200), (200, 640)]
    gen = torch.Generator().manual_seed(3)
    Ws = [torch.rand(s, generator=gen) - 0.5 for s in shapes]
    Gs = [torch.randn(s, generator=gen) for s in shapes]
    Ms = [torch.randn(s, generator=gen) for s in shapes]
    dm.dmuon_set_wait_timeout(handle.h, 1)
    dm.dmuon_set_fused_phases(handle.h, fused)
    try:
        handle.step(_to_dev(Ws), _to_dev(Gs), _to_dev(Ms))
        rc, _ = handle.status(2)
    finally:
        dm.dmuon_set_wait_timeout(handle.h, 0)
        dm.dmuon_set_fused_phases(handle.h, 2)
    assert rc == -6
    assert handle.status(2)[0] == 0   # the error word was cleared by the read
    _step_and_check(handle, Ws, Gs, Ms)


@pytest.mark.parametrize("fused", [True, False])
def test_launch_count_and_profile(handle, fused):
    shapes = [(256, 512), (512, 256)]
    Ws = [torch.zeros(s, device="cuda") for s in shapes]
    Gs = [torch.randn(s, device="cuda") for s in shapes]
    Ms = [torch.zeros(s, device="cuda") for s in shapes]
    dm.dmuon_set_fused_phases(handle.h, fused)
    try:
        dm.dmuon_profile_enable(handle.h, True)
        dm.dmuon_profile_read(handle.h)
        before = dm.dmuon_launch_count(handle.h)
        handle.step(Ws, Gs, Ms, ns_steps=5)
        assert dm.dmuon_launch_count(handle.h) - before == (4 + 1 if fused else 4 + 3 * 5)
        prof = dm.dmuon_profile_read(handle.h)
        dm.dmuon_profile_enable(handle.h, False)
    finally:
        dm.dmuon_set_fused_phases(handle.h, 2)
    # the momentum kernel runs twice (the pass and the prescale redo pass), as does the finalisation
    assert prof["momentum"][1] == 2 and prof["finalize"][1] == 2
    if fused:
        assert prof["ns_fused"][1] == 1 and prof["gram"][1] == 0 and prof["apply"][1] == 0
    else:
        assert prof["gram"][1] == 5 and prof["apply"][1] == 5 and prof["ns_fused"][1] == 0
    assert all(v[0] >= 0 for v in prof.values())
    assert "matrices 2" in dm.dmuon_plan_summary(handle.h)
    assert handle.status()[0] == 0


@pytest.mark.parametrize("tiles", [1, 2, 3])
def test_fused_phases_bitwise_equal_per_phase_launches(tiles):
    """One fused launch per chunk runs the same tiles with the same
    arithmetic as one launch per phase and iteration: weights and momenta
    bitwise equal, on single CTAs and CTA pairs, for a list mixing shapes
    (k/v-like short sides, tall and wide, ragged), over two chunks, with the
    weight update, a standalone Newton-Schulz call and 1, 2 and 7 steps."""
    gen = torch.Generator().manual_seed(53)
    shapes = [(300, 700), (700, 300), (1024, 256), (257, 1100), (512, 512), (130, 2000), (96, 640)]
    Ws = [torch.rand(s, generator=gen) - 0.5 for s in shapes]
    Gs = [torch.randn(s, generator=gen) for s in shapes]
    Ms = [torch.randn(s, generator=gen) for s in shapes]
    res = {}
    for fused in (True, False):
        with dm.Handle(0) as h2:
            dm.dmuon_set_tile_mode(h2.h, tiles)
            dm.dmuon_set_small_path(h2.h, False)
            dm.dmuon_set_chunk_elements(h2.h, 700_000)
            dm.dmuon_set_fused_phases(h2.h, fused)
            out = []
            for ns in (5, 1, 2, 7):
                Wd, Gd, Md = _to_dev(Ws), _to_dev(Gs), _to_dev(Ms)
                h2.step(Wd, Gd, Md, ns_steps=ns)
                assert h2.status()[0] == 0
                out += [x.cpu() for x in Wd + Md]
            O = [torch.empty(s, device="cuda") for s in shapes]
            h2.newton_schulz(_to_dev(Gs), O)
            assert h2.status()[0] == 0
            out += [o.cpu() for o in O]
            assert "chunks 3 " in dm.dmuon_plan_summary(h2.h)
            res[fused] = out
    for a, b in zip(res[True], res[False]):
        assert torch.equal(a, b)
    with dm.Handle(0) as h3:   # and the fused launch against the oracle
        dm.dmuon_set_tile_mode(h3.h, tiles)
        dm.dmuon_set_small_path(h3.h, False)
        dm.dmuon_set_chunk_elements(h3.h, 700_000)
        _step_and_check(h3, Ws, Gs, Ms)


# ---------------------------------------------------------------- full size

def _full_size_sampled(handle, name, sample, steps_before=None):
    """Run the whole workload (bench launch configuration) on the GPU with
    seeded device inputs; compare the sampled matrices' last-step update and
    momentum with the oracle run from the same seeded inputs."""
    w = workloads.get(name)
    n = len(w.shapes)
    warm = w.warm_steps if steps_before is None else steps_before
    dev = "cuda"
    Wd = [workloads.weight(w, i, dev) for i in range(n)]
    Md = [workloads.momentum(w, i, dev) for i in range(n)]
    for step in range(warm):
        Gd = [workloads.grad(w, i, step, dev) for i in range(n)]
        handle.step(Wd, Gd, Md)
        del Gd
    Gd = [workloads.grad(w, i, warm, dev) for i in range(n)]
    W_before = {i: Wd[i].cpu() for i in sample}
    handle.step(Wd, Gd, Md)
    rc, _ = handle.status()
    assert rc == 0
    for i in sample:
        # momentum history from the seeded inputs alone
        M = workloads.momentum(w, i, dev).cpu().numpy().astype(np.float64)
        for step in range(warm):
            M = oracle.momentum_update(M, workloads.grad(w, i, step, dev).cpu().numpy(), F32(0.95))
            M = M.astype(np.float32).astype(np.float64)  # the fp32 state between steps
        G = Gd[i].cpu().numpy()
        r, c = w.shapes[i]
        ref = oracle.muon_step(np.zeros((r, c)), G, M, lr=F32(0.02), mu=F32(0.95))
        upd = Wd[i].cpu().numpy().astype(np.float64) - W_before[i].numpy().astype(np.float64)
        assert_momentum(Md[i].cpu().numpy(), ref["M"], "%s matrix %d" % (name, i))
        e_u = rel_fro(upd, ref["W"])
        assert e_u <= NS_TOL, (name, i, w.shapes[i], e_u)
    del Wd, Md, Gd
    torch.cuda.empty_cache()


@pytest.mark.slow
def test_full_llama3_8b_sampled(handle):
    # layer 0: q, k, v, gate (transposed path), down; layer 31: k
    _full_size_sampled(handle, "llama3_8b", [0, 1, 2, 4, 6, 218])


@pytest.mark.slow
def test_full_spiked_4096_sampled(handle):
    _full_size_sampled(handle, "spiked_4096", [0, 63])


@pytest.mark.slow
def test_full_tp_70b_mixed_sampled(handle):
    # the 28672x8192 matrix (transposed, short side 8192) and four 64x256 ones
    _full_size_sampled(handle, "tp_70b_mixed", [0, 1, 2, 256, 512])


@pytest.mark.slow
@pytest.mark.parametrize("shape", [(32768, 32768), (65536, 32768)])
@pytest.mark.parametrize("backend", ["direct", "gram"])
def test_max_short_side_signed_permutation(handle, shape, backend):
    """Short side at the limit (DMUON_MAX_SHORT_SIDE = 32768): G = alpha * P
    with P a signed permutation (one +-1 per column of the oriented matrix)
    and alpha a power of two, so every bf16 rounding of the input is exact.
    All singular values of the normalised input equal
    sigma = alpha / (alpha sqrt(m) + eps), hence O = p(sigma) P with p the
    composed scalar quintic, taken from the oracle's direct iteration on
    the 1x1 matrix [sigma]."""
    r, c = shape
    m = min(r, c)
    alpha = 2.0 ** -10
    gen = torch.Generator(device="cuda").manual_seed(77)
    perm = torch.randperm(max(r, c), generator=gen, device="cuda")[:m]
    sign = torch.randint(0, 2, (m,), generator=gen, device="cuda").float() * 2 - 1
    G = torch.zeros(shape, device="cuda")
    idx = torch.arange(m, device="cuda")
    if r <= c:
        G[idx, perm] = alpha * sign
    else:
        G[perm, idx] = alpha * sign
    O = torch.empty_like(G)
    with dm.Handle(0) as h2:
        if backend == "gram":   # the printed table, as the expected value below
            h2.gram_newton_schulz([G], [O], coeffs=oracle.coefficient_rows(5))
        else:
            h2.newton_schulz([G], [O])
        assert h2.status()[0] == 0
        assert "backend %s" % backend in dm.dmuon_plan_summary(h2.h)
    sigma = alpha / (alpha * np.sqrt(m) + 1e-7)
    p_sigma = float(oracle.newton_schulz_direct(np.array([[sigma]]), oracle.coefficient_rows(5))[0, 0])
    expect_vals = p_sigma * sign
    got_vals = O[idx, perm] if r <= c else O[perm, idx]
    # the nonzero pattern: everything off the permutation is (close to) zero
    tot = float((O * O).sum(dtype=torch.float64))
    on = float((got_vals * got_vals).sum(dtype=torch.float64))
    assert tot - on <= 1e-4 * tot, (tot, on)
    diff = got_vals - expect_vals
    err = float(torch.sqrt((diff * diff).sum(dtype=torch.float64) / (expect_vals * expect_vals).sum(dtype=torch.float64)))
    assert err <= NS_TOL, (shape, backend, p_sigma, err)
    del G, O
    torch.cuda.empty_cache()


@pytest.mark.parametrize("backend", ["direct", "gram"])
def test_max_long_side(handle, backend):
    """Long side at DMUON_MAX_DIM = 2^20 (8 x 2^20 and its transpose): one
    super-tile whose X X^T runs 16384 K blocks, 4096 column tiles in the
    Apply phase; against the fp64 oracle directly."""
    gen = torch.Generator().manual_seed(91)
    shapes = [(8, 1 << 20), (1 << 20, 8)]
    ins = [torch.randn(s, generator=gen) for s in shapes]
    outs = [torch.empty(s, device="cuda") for s in shapes]
    if backend == "gram":   # the printed table on both backends (the Gram default is Polar Express)
        handle.gram_newton_schulz(_to_dev(ins), outs, coeffs=oracle.coefficient_rows(5))
    else:
        handle.newton_schulz(_to_dev(ins), outs)
    assert handle.status()[0] == 0
    for x, o, s in zip(ins, outs, shapes):
        e = rel_fro(o.cpu().numpy(), oracle.newton_schulz(x.numpy()))
        assert e <= NS_TOL, (s, backend, e)


@pytest.mark.parametrize("backend,chunk", [("direct", 0), ("direct", 300_000), ("gram", 0), ("gram", 300_000)])
def test_random_shape_lists(handle, backend, chunk):
    """40 seeded random shapes (1..700 per side) in one call: small-kernel,
    explicit- and implicit-restart matrices interleaved in the caller's list,
    so plan ordering, pointer permutation and chunk boundaries all take
    part; every matrix against the fp64 oracle (direct or Gram)."""
    from oracle import gram as og
    rng = np.random.default_rng(20261202)
    shapes = [tuple(int(v) for v in rng.integers(1, 701, size=2)) for _ in range(40)]
    shapes[3] = (64, 256)
    shapes[7] = (700, 64)   # n >= 2m
    shapes[11] = (400, 400)
    gen = torch.Generator().manual_seed(5)
    Ws = [torch.rand(s, generator=gen) - 0.5 for s in shapes]
    Gs = [torch.randn(s, generator=gen) for s in shapes]
    Ms = [torch.randn(s, generator=gen) for s in shapes]
    Wd, Gd, Md = _to_dev(Ws), _to_dev(Gs), _to_dev(Ms)
    with dm.Handle(0) as h2:
        if chunk:
            dm.dmuon_set_chunk_elements(h2.h, chunk)
        h2.step(Wd, Gd, Md, lr=0.05, mu=0.9, backend=backend)
        rc, flags = h2.status(len(shapes))
        assert rc == 0 and not any(flags)
    step = og.muon_step_gram if backend == "gram" else oracle.muon_step
    for i, s in enumerate(shapes):
        ref = step(Ws[i].numpy(), Gs[i].numpy(), Ms[i].numpy(), lr=F32(0.05), mu=F32(0.9))
        W0 = Ws[i].numpy().astype(np.float64)
        assert_momentum(Md[i].cpu().numpy(), ref["M"], "matrix %d %s" % (i, s))
        e = rel_fro(Wd[i].cpu().numpy().astype(np.float64) - W0, ref["W"] - W0)
        assert e <= NS_TOL, (i, s, backend, chunk, e)

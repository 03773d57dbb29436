"""Host-side checks of the C ABI (no GPU needed).

The library must build for sm_103a, load, and export every function that
include/dmuon.h declares; the host-only entry points (defaults, workspace
sizing, error strings) and the argument checks that run before any device
work are exercised here.  Compute calls are left to the gpu-marked tests.
"""
import ctypes
import os
import re

import pytest

import newton_schulz_nesterov_gb300 as dm
import oracle
from newton_schulz_nesterov_gb300 import _build, flops, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return dm.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "dmuon.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dmuon_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("dmuon_create", "dmuon_destroy", "dmuon_step", "dmuon_newton_schulz",
                 "dmuon_get_status", "dmuon_workspace_bytes", "dmuon_error_string"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_version_and_error_strings(lib):
    assert "sm_103a" in dm.dmuon_version()
    for code in dm.STATUS:
        s = dm.dmuon_error_string(code)
        assert s and s != "unknown status"
    assert dm.dmuon_error_string(12345) == "unknown status"


def test_default_opts_are_the_pages_defaults(lib, golden_dir):
    gold = {}
    for line in open(os.path.join(golden_dir, "muon_defaults.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            gold[k] = float(v)
    o = dm.Opts()
    o.eps = -1.0
    o.nesterov = 7
    lib.dmuon_default_opts(ctypes.byref(o))
    assert o.weight_decay == gold["weight_decay"]
    assert o.eps == pytest.approx(gold["eps"], rel=1e-7)
    assert o.nesterov == int(gold["nesterov"])
    assert o.scale_mode == 0
    assert not o.coeffs
    lib.dmuon_default_opts(None)  # no-op, no crash


def _chunks(shapes, limit=1 << 29):
    """Greedy contiguous chunks of at most `limit` elements (the library's rule)."""
    out, cur, tot = [], [], 0
    for s in shapes:
        e = s[0] * s[1]
        if cur and tot + e > limit:
            out.append(cur)
            cur, tot = [], 0
        cur.append(s)
        tot += e
    if cur:
        out.append(cur)
    return out


def test_workspace_bytes_covers_the_largest_chunk(lib):
    for name in ("tinymlp_d128", "tinymlp_d512", "llama3_8b", "tp_70b_mixed", "spiked_4096"):
        shapes = list(workloads.get(name).shapes)
        got = dm.dmuon_workspace_bytes(shapes)
        per = lambda ch: sum(2 * (2 * min(r, c) * max(r, c) + 2 * min(r, c) ** 2) for r, c in ch)  # noqa: E731
        need = max(per(ch) for ch in _chunks(shapes))
        assert need <= got <= need * 1.05 + 64 * 1024 * 1024, (name, need, got)
    # the Llama set needs a few layers' worth, not all 224 matrices at once
    llama = list(workloads.get("llama3_8b").shapes)
    assert dm.dmuon_workspace_bytes(llama) < 4e9
    assert len(_chunks(llama)) == 14
    assert dm.dmuon_workspace_bytes([]) == 0


def test_workspace_bytes_rejects_bad_shapes(lib):
    for bad in ([(0, 4)], [(4, -1)], [(1 << 21, 8)], [(40000, 40000)]):
        with pytest.raises(dm.DmuonError) as e:
            dm.dmuon_workspace_bytes(bad)
        assert e.value.code == -1
    out = ctypes.c_size_t()
    assert lib.dmuon_workspace_bytes(None, -1, ctypes.byref(out)) == -1
    assert lib.dmuon_workspace_bytes(None, 3, ctypes.byref(out)) == -1
    assert lib.dmuon_workspace_bytes(None, 0, None) == -1


def test_null_handle_is_rejected(lib):
    assert lib.dmuon_step(None, None, None, None, None, 0, 0.02, 0.95, 5, None, None) == -1
    assert lib.dmuon_newton_schulz(None, None, None, None, 1, 5, None, 1e-7, None) == -1
    assert lib.dmuon_get_status(None, None, 0) == -1
    assert lib.dmuon_launch_count(None) == -1
    assert lib.dmuon_profile_enable(None, 1) == -1
    assert lib.dmuon_set_wait_timeout(None, 5) == -1
    assert lib.dmuon_set_small_path(None, 1) == -1
    assert lib.dmuon_set_balanced_dealing(None, 1) == -1
    assert lib.dmuon_gram_newton_schulz(None, None, None, None, 1, 5, None, None, 0, 1e-7, None) == -1
    assert lib.dmuon_last_error(None) == b"null handle"
    assert lib.dmuon_plan_summary(None, None, 0) == -1
    lib.dmuon_destroy(None)


def test_create_without_a_gpu_fails_cleanly(lib):
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except ImportError:
        pass
    h = ctypes.c_void_p(1)
    rc = lib.dmuon_create(ctypes.byref(h), 0)
    assert rc in (-1, -4, -7)
    assert not h.value
    assert lib.dmuon_create(None, 0) == -1


def test_workload_shapes_and_flop_totals():
    """Shape lists and the algorithmic / dense FLOP totals of each workload
    (totals computed by hand from the shape lists)."""
    w1 = workloads.get("tinymlp_d128").shapes
    assert len(w1) == 12 and w1.count((512, 128)) == 8 and w1.count((128, 512)) == 4
    w3 = workloads.get("llama3_8b").shapes
    assert len(w3) == 224 and sum(r * c for r, c in w3) == 6979321856
    w5 = workloads.get("tp_70b_mixed").shapes
    assert len(w5) == 513 and w5[0] == (28672, 8192)
    # 5*(3 m^2 n + m^3), one TinyMLP-128 matrix: m=128, n=512
    assert flops.algorithmic_flops([(512, 128)]) == 5 * (3 * 128 * 128 * 512 + 128 ** 3)
    assert flops.algorithmic_flops(w1) == 1_635_778_560
    assert round(flops.algorithmic_flops(w3) / 1e12, 1) == 471.8
    assert round(flops.dense_flops(w3) / 1e12, 1) == 665.9
    assert round(flops.algorithmic_flops(workloads.get("spiked_4096").shapes) / 1e12, 1) == 88.0
    assert round(flops.algorithmic_flops(w5) / 1e12, 1) == 31.6


def test_gram_flop_count():
    """Gram backend: per window X X^T (m^2 n) and Q X (2 m^2 n), Z (m^3 per
    step), Q' (m^3, not on the window's first step), R Z and Z (R Z) (2 m^3,
    not on its last); windows longer than two steps are split."""
    m, n = 96, 150
    assert flops.gram_windows(5, (2,)) == flops.gram_windows(5, ()) == [(0, 2), (2, 4), (4, 5)]
    assert flops.gram_flops([(m, n)]) == 9 * m * m * n + 11 * m ** 3
    assert flops.gram_flops([(n, m)], 5, ()) == flops.gram_flops([(n, m)], 5, (2, 4))
    assert flops.gram_flops([(m, n)], 1, (2,)) == 3 * m * m * n + m ** 3      # one window, one step
    assert flops.gram_flops([(m, n)], 2, ()) == 3 * m * m * n + 5 * m ** 3    # Z, W, R', Z, Q'
    assert flops.gram_flops([(m, n)], 3, (1, 2)) == 3 * (3 * m * m * n + m ** 3)
    assert flops.gram_flops([(m, n)], 0) == 0
    assert flops.gram_windows(8, ()) == [(0, 2), (2, 4), (4, 6), (6, 8)]
    assert flops.gram_windows(7, (2, 4)) == [(0, 2), (2, 4), (4, 6), (6, 7)]
    assert flops.gram_windows(5, (1,)) == [(0, 1), (1, 3), (3, 5)]
    # 9 m^2 n + 11 m^3 against 15 m^2 n + 5 m^3: cheaper when n > m, equal for square matrices
    assert flops.gram_flops([(1024, 4096)]) < flops.algorithmic_flops([(1024, 4096)])
    assert flops.gram_flops([(1024, 1024)]) == flops.algorithmic_flops([(1024, 1024)])  # break-even at n = m


def test_gram_workspace_bytes(lib):
    shapes = list(workloads.get("llama3_8b").shapes)
    direct = dm.dmuon_workspace_bytes(shapes)
    gram = dm.dmuon_workspace_bytes(shapes, "gram")
    # chunks hold eight m x m fp16 buffers per matrix in place of A and B
    assert direct < gram < 4 * direct
    out = ctypes.c_size_t()
    arr = (dm.Shape * 1)(dm.Shape(64, 64))
    assert lib.dmuon_workspace_bytes_ex(arr, 1, 7, ctypes.byref(out)) == -1
    assert lib.dmuon_workspace_bytes_ex(arr, 1, 0, ctypes.byref(out)) == 0
    assert lib.dmuon_workspace_bytes_ex(arr, 1, 1, ctypes.byref(out)) == 0 and out.value > 0


def test_inputs_are_seeded_and_shaped():
    torch = pytest.importorskip("torch")
    w = workloads.get("tinymlp_d128")
    a = workloads.grad(w, 2, 0)
    b = workloads.grad(w, 2, 0)
    c = workloads.grad(w, 2, 1)
    assert a.shape == (128, 512) and a.dtype == torch.float32
    assert torch.equal(a, b) and not torch.equal(a, c)
    W = workloads.weight(w, 0)
    assert float(W.abs().max()) <= 1.0 / 128 ** 0.5
    s = workloads.get("spiked_4096")
    # rank-16 spike on a small stand-in shape: top singular value near 1e2
    small = workloads.Workload("s", ((256, 256),), 0.0, "zero", 0, spike_rank=16)
    g = workloads.grad(small, 0)
    sv = torch.linalg.svdvals(g.double())
    assert abs(float(sv[0]) - 100.0) < 1e-3 and abs(float(sv[15]) - 1e-3) < 1e-5
    assert s.spike_rank == 16


def test_polar_express_table_matches_the_oracle(lib):
    """The library's Polar Express construction (its own Remez exchange, in
    C++) against the oracle's (numpy), for the default start and others."""
    import numpy as np
    from oracle import polar_express as pe
    for steps, lo, hi, s in [(5, 1e-3, 1.0, 1.05), (8, 1e-3, 1.0, 1.05), (5, 1e-2, 1.0, 1.0),
                             (3, 0.1, 1.5, 1.02), (1, 0.5, 1.0, 1.05)]:
        got = np.array(dm.dmuon_polar_express_coefficients(steps, lo, hi, s))
        ref = np.array(pe.polar_express_rows(steps, lo, hi, s))
        assert got.shape == (steps, 3)
        assert np.max(np.abs(got - ref) / np.abs(ref)) <= 1e-6, (steps, lo, hi, s)


def test_polar_express_argument_errors(lib):
    out = (ctypes.c_float * 3)()
    f = lib.dmuon_polar_express_coefficients
    assert f(0, 1e-3, 1.0, 1.05, out) == -1
    assert f(65, 1e-3, 1.0, 1.05, out) == -1
    assert f(1, 0.0, 1.0, 1.05, out) == -1
    assert f(1, 1.0, 1.0, 1.05, out) == -1
    assert f(1, 1e-3, 1.0, 0.0, out) == -1
    assert f(1, 1e-3, 1.0, 1.05, None) == -1
    assert f(1, 1e-3, 1.0, 1.05, out) == 0


def test_gram_range_check(lib):
    """The Gram backend's fp16 range check: the default and the Polar Express
    tables fit (the latter's first row, a ~ 8, b ~ -22, c ~ 15, is far past
    the crude |a| + 2|b| + 4|c| <= 40 rule yet keeps every buffer small);
    tables that could overflow a buffer are refused with the reason."""
    ok, why = dm.dmuon_gram_check_coefficients(5)
    assert ok and why == ""
    assert dm.dmuon_gram_check_coefficients(5, dm.dmuon_polar_express_coefficients(5))[0]
    assert dm.dmuon_gram_check_coefficients(5, dm.dmuon_polar_express_coefficients(5), restarts=())[0]
    # eight steps without restarts run as four windows of two steps
    assert dm.dmuon_gram_check_coefficients(8, restarts=())[0]
    assert dm.dmuon_gram_check_coefficients(8, oracle.coefficient_rows(8), restarts=())[0]
    assert dm.dmuon_gram_check_coefficients(8, restarts=(3, 6))[0]
    ok, why = dm.dmuon_gram_check_coefficients(1, [(1.0, 100.0, 0.0)])
    assert not ok and "kappa R Z" in why     # 1024 x 101 at the top of the spectrum
    ok, why = dm.dmuon_gram_check_coefficients(3, [(1.0, 25.0, 0.0)] * 3, restarts=())
    assert not ok and "singular values" in why   # x + 25 x^3 sends 1 to 26
    for row in ((0.0, 1.0, 0.0), (0.0, 0.0, 1.0), (-1.0, 2.0, 0.0), (0.01, 1.0, 0.0)):
        ok, why = dm.dmuon_gram_check_coefficients(1, [row])
        assert not ok and "1/64" in why          # no identity part: the fp16 Z would lose its small entries
    assert dm.dmuon_gram_check_coefficients(1, [(1.0 / 64, 1.0, 0.0)])[0]
    ok, _ = dm.dmuon_gram_check_coefficients(0)
    assert ok
    # argument errors
    assert lib.dmuon_gram_check_coefficients(-1, None, None, 0, None, 0) == -1
    assert lib.dmuon_gram_check_coefficients(65, None, None, 0, None, 0) == -1
    assert lib.dmuon_gram_check_coefficients(5, None, None, 2, None, 0) == -1
    nan = (ctypes.c_float * 3)(float("nan"), 0.0, 0.0)
    assert lib.dmuon_gram_check_coefficients(1, nan, None, 0, None, 0) == -1


def _preview(shapes, **kw):
    out = dm.dmuon_plan_preview(shapes, **kw)
    fields = dict(part.strip().split(" ", 1) for part in out.split(";"))
    bal = fields["balance"].split()
    items = fields["items"].split()
    return out, {"tiles": fields["tiles"], "chunks": int(fields["chunks"].split()[0]),
                 "small": int(fields["small-matrix"].split()[-1]),
                 "items": {items[i]: int(items[i + 1]) for i in range(0, 6, 2)},
                 "balance": {bal[i]: float(bal[i + 1]) for i in range(0, 6, 2)}}


def _pair_items(shapes):
    """Work items of a CTA-pair plan counted from their definition: upper
    256 x 256 super-tiles for the symmetric phases, all 256 x 256 output
    tiles of the m x n iterate for the apply phase."""
    cd = lambda a, b: -(-a // b)  # noqa: E731
    g = a = 0
    for r, c in shapes:
        m, n = min(r, c), max(r, c)
        T = cd(m, 256)
        g += T * (T + 1) // 2
        a += T * cd(n, 256)
    return {"gram": g, "gram2": g, "apply": a}


def test_plan_preview_items_dealing_and_chunks(lib):
    """The host planner without a device: work-item counts match their
    definition, longest-first dealing evens one Llama-3-8B layer's Gram list
    (strided leaves the pairs that drew extra long tiles ~10 % behind), the
    full set splits into 14 chunks of at most 2^29 elements, for either
    backend."""
    layer = workloads.get("llama3_8b_1layer").shapes
    _, p = _preview(layer)
    assert p["tiles"] == "256x256 CTA pairs" and p["chunks"] == 1
    assert p["items"] == _pair_items(layer)
    assert p["balance"]["gram"] <= 1.02 and p["balance"]["apply"] <= 1.01
    _, q = _preview(layer, balanced=False)
    assert q["items"] == p["items"] and q["balance"]["gram"] >= 1.08
    full = workloads.get("llama3_8b").shapes
    _, f = _preview(full)
    assert f["chunks"] == 14 and f["items"] == _pair_items(full) and f["balance"]["gram"] <= 1.02
    _, gb = _preview(full, backend="gram")
    assert gb["chunks"] == 14 and gb["items"] == _pair_items(full)


def _narrow_items(shapes):
    """Work items of a 128 x 128 single-CTA plan from their definition: blocks
    (I, J), I <= J, of the m x m products; all 128 x 128 output tiles of the
    m x n iterate for the apply phase."""
    cd = lambda a, b: -(-a // b)  # noqa: E731
    g = a = 0
    for r, c in shapes:
        m, n = min(r, c), max(r, c)
        T = cd(m, 128)
        g += T * (T + 1) // 2
        a += T * cd(n, 128)
    return {"gram": g, "gram2": g, "apply": a}


def test_plan_preview_tile_choice(lib):
    """Automatic tiles: CTA pairs only when some chunked matrix's short side
    exceeds 128 and there is at least one Gram super-tile per pair; small
    matrices go to the small-matrix kernel and do not count.  Single CTAs
    take 128 x 128 tiles when the 128 x 256 Gram items would not cover the
    SMs, else 128 x 256."""
    d512 = workloads.get("tinymlp_d512").shapes            # 12 x 3 = 36 super-tiles
    out, p = _preview(d512)                                 # 36 < 76 pairs; 72 halves < 152 SMs
    assert p["tiles"] == "128x128 single CTAs" and p["items"] == _narrow_items(d512)
    assert p["items"] == {"gram": 120, "gram2": 120, "apply": 768}
    assert "CTA pairs" in _preview(d512, clusters=36)[0]
    assert "128x128 single CTAs" in _preview(d512, clusters=37)[0]
    assert "128x256 single CTAs" in _preview(d512, tile_mode=1)[0]
    assert "128x128 single CTAs" in _preview(d512, tile_mode=3)[0]
    assert "128x256 single CTAs" in _preview(d512, sms=72)[0]           # 72 halves cover 72 SMs
    assert "128x128 single CTAs" in _preview(d512, sms=73)[0]
    assert "CTA pairs" in _preview(d512, tile_mode=2)[0]
    assert "128x256 single CTAs" in _preview(workloads.get("llama3_8b_1layer").shapes, tile_mode=1)[0]
    assert "128x128 single CTAs" in _preview(workloads.get("llama3_8b_1layer").shapes, tile_mode=3)[0]
    assert "single CTAs" in _preview(d512, clusters=0, tile_mode=0)[0]
    assert "128x256 single CTAs" in _preview(list(d512) * 4, clusters=0)[0]   # 288 halves >= 152
    _, s = _preview(workloads.get("tinymlp_d128").shapes)
    assert s["small"] == 12 and s["chunks"] == 0
    _, t = _preview(workloads.get("tp_70b_mixed").shapes)
    assert t["small"] == 512 and t["tiles"] == "256x256 CTA pairs" and t["items"]["gram"] == 32 * 33 // 2
    assert "backend gram; tiles 256x256 CTA pairs" in _preview(d512, backend="gram")[0]


def test_plan_preview_argument_errors(lib):
    sh = (dm.Shape * 1)()
    sh[0].rows, sh[0].cols = 64, 64
    f = lib.dmuon_plan_preview
    assert f(sh, 1, 1, 0, 0, 152, 1, None, 0) == -1      # Gram backend without clusters
    assert f(sh, 1, 7, 0, 76, 152, 1, None, 0) == -1     # unknown backend
    assert f(sh, 1, 0, 4, 76, 152, 1, None, 0) == -1     # unknown tile mode
    assert f(sh, 1, 0, 0, 76, 0, 1, None, 0) == -1       # no SMs
    assert f(None, 1, 0, 0, 76, 152, 1, None, 0) == -1
    sh[0].rows = 0
    assert f(sh, 1, 0, 0, 76, 152, 1, None, 0) == -1     # empty matrix
    assert f(None, 0, 0, 0, 76, 152, 1, None, 0) > 0     # an empty list previews an empty plan


def _gram_buffer_peaks(X, rows, restarts, kappa=1024.0):
    """Largest magnitudes the Gram-space buffers reach for input X (fp64,
    unrounded): kappa R, kappa R Z, Z, each window's factor and the product
    of the window factors, following the Gram iteration's algebra."""
    import numpy as np
    m = X.shape[0]
    eye = np.eye(m)
    cuts = sorted({k for k in restarts if 0 < k < len(rows)})
    bounds = [0] + cuts + [len(rows)]
    peak = dict(kR=0.0, kRZ=0.0, Z=0.0, Q=0.0, total=0.0)
    acc = eye
    for s, e in zip(bounds, bounds[1:]):
        R = X @ X.T
        Q = eye
        for a, b, c in rows[s:e]:
            peak["kR"] = max(peak["kR"], kappa * np.abs(R).max())
            Z = a * eye + b * R + c * R @ R
            peak["Z"] = max(peak["Z"], np.abs(Z).max())
            peak["kRZ"] = max(peak["kRZ"], kappa * np.abs(R @ Z).max())
            Q = Z @ Q
            peak["Q"] = max(peak["Q"], np.abs(Q).max())
            R = Z @ R @ Z
        acc = Q @ acc
        peak["total"] = max(peak["total"], np.abs(acc).max())
        X = Q @ X
    return peak


def test_gram_range_check_is_sound(lib):
    """Every table the fp16 range check accepts keeps each Gram-space buffer
    within the limits it promises (kappa R, kappa R Z and Z under 32768, a
    window's factor under 8192, the accumulated factor under 32768) on inputs
    built to reach each polynomial's extremes: singular values at 1, at the
    points where |p| peaks, spread over (0, 1], and random ones."""
    import numpy as np
    rng = np.random.default_rng(31)
    tables = [(None, (2,)), (dm.dmuon_polar_express_coefficients(5), (2,)),
              (dm.dmuon_polar_express_coefficients(5), ()), ([(1.0, 20.0, 0.0)], ()), ([(3.0, -8.0, 6.0)] * 3, (1,))]
    restart_sets = [(), (2,), (1, 3)]
    you = [(4.0848, -6.8946, 2.927), (3.9505, -6.3029, 2.6377), (3.7418, -5.5913, 2.3037),
           (2.8769, -3.1427, 1.2046), (2.8366, -3.0525, 1.2012)]
    for _ in range(8):   # Newton-Schulz-like tables: the default rows perturbed by ~15 %
        tables.append(([tuple(v * (1 + 0.15 * rng.standard_normal()) for v in r) for r in you],
                       restart_sets[int(rng.integers(3))]))
    checked = 0
    for coeffs, restarts in tables:
        steps = 5 if coeffs is None else len(coeffs)
        ok, _ = dm.dmuon_gram_check_coefficients(steps, coeffs, restarts=restarts)
        if not ok:
            continue
        checked += 1
        rows = [tuple(float(v) for v in r) for r in (coeffs or [(4.0848, -6.8946, 2.927), (3.9505, -6.3029, 2.6377),
                                                                 (3.7418, -5.5913, 2.3037), (2.8769, -3.1427, 1.2046),
                                                                 (2.8366, -3.0525, 1.2012)])]
        # singular values: 1, where the first step's |p| peaks on (0, 1], a spread, random
        a, b, c = rows[0]
        crit = [x for x in np.sqrt(np.roots([5 * c, 3 * b, a]).real.clip(0)) if 0 < x <= 1] if c else []
        spectra = [np.ones(8), np.array(crit + [1.0] * (8 - len(crit))), np.linspace(0.05, 1, 8), rng.uniform(0, 1, 8)]
        for sv in spectra:
            U, _ = np.linalg.qr(rng.standard_normal((8, 8)))
            V, _ = np.linalg.qr(rng.standard_normal((20, 8)))
            X = (U * (sv / max(1.0, sv.max()))) @ V.T          # spectral norm <= 1
            p = _gram_buffer_peaks(X, rows, restarts)
            assert p["kR"] <= 32768 and p["kRZ"] <= 32768 and p["Z"] <= 32768, (rows, restarts, p)
            assert p["Q"] <= 8192 and p["total"] <= 32768, (rows, restarts, p)
    assert checked >= 6   # the perturbed tables that let singular values run past ~1.3 are refused


def test_bench_fused_roofline_arithmetic():
    """The fused kernel's roofline object from made-up timings: all of the
    chunked matrices' algorithmic flops over the kernel's time, and per
    launch the algorithmic bytes of every product of a chunk."""
    import bench
    shapes = [(4096, 4096), (1024, 4096), (64, 256)]        # the last goes to the small-matrix kernel
    r = bench.fused_roofline(shapes, steps=2, fused_ms=40.0, fused_n=4, peak=1000.0, peak_src="x",
                             pairs=True, launch_traffic=7e9)
    fl = 5 * (3 * 4096 ** 3 + 4096 ** 3) + 5 * (3 * 1024 ** 2 * 4096 + 1024 ** 3)
    assert r["achieved"] == pytest.approx(fl * 2 / 0.040 / 1e12)
    assert r["launches_per_step"] == 2 and r["avg_launch_ms"] == 10.0
    per_iter = 2 * (3 * 4096 * 4096 + 4 * 4096 ** 2) + 2 * (3 * 1024 * 4096 + 4 * 1024 ** 2)
    assert r["algorithmic_bytes"] == pytest.approx(per_iter * 5 / 2)
    assert r["traffic"] == 7e9 and "Fused" in r["kernel"]
    assert bench.fused_traffic("tinymlp_d128") is None


def test_bench_apply_roofline_arithmetic():
    """bench.py's roofline object from made-up timings: achieved rate, the
    per-launch traffic and algorithmic bytes follow from the shapes."""
    import bench
    shapes = [(4096, 4096), (1024, 4096), (64, 256)]        # the last goes to the small-matrix kernel
    r = bench.apply_roofline(shapes, steps=2, apply_ms=10.0, apply_n=10, peak=1000.0, peak_src="x",
                             pairs=True, step_traffic=5e9)
    fl = 5 * 2 * (4096 ** 3 + 1024 ** 2 * 4096)             # 2 m^2 n per iteration, 5 iterations
    assert r["achieved"] == pytest.approx(fl * 2 / 0.010 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / 1000.0)
    assert r["launches_per_step"] == 5 and r["avg_launch_ms"] == 1.0
    alg = 2 * (2 * 4096 * 4096 + 4096 ** 2) + 2 * (2 * 1024 * 4096 + 1024 ** 2)
    assert r["algorithmic_bytes"] == pytest.approx(alg * 5 / 5)
    assert r["traffic"] == pytest.approx(5e9 * 5 / 5)
    assert "CTA-pair" in r["kernel"] and r["bound"] == "tensor"
    assert bench.apply_roofline(shapes, 1, 1.0, 5, 1.0, "x", False, None)["traffic"] is None

"""Allocation-free Newton-Schulz entry point (collected last on purpose).

dmuon_newton_schulz_noalloc serves callers that may not call cudaMalloc: a
host framework that owns all device memory, a plugin handed only its input
and output buffers, or a path that cannot take cudaMalloc's implicit
synchronisation.  Its scratch is a static device array shared by all calls.
This test calls it through the C ABI twice in a row, on two different
shapes so that the second call would expose any leftover of the first, and
compares each output with the handle-based dmuon_newton_schulz output within
the parity tolerance (relative Frobenius error 3e-2).  It must pass alone in
a fresh process and after the rest of the suite.
"""
import ctypes

import pytest

torch = pytest.importorskip("torch")

import newton_schulz_nesterov_gb300 as dm  # noqa: E402
from newton_schulz_nesterov_gb300 import _build  # noqa: E402

pytestmark = pytest.mark.gpu

NS_TOL = 3e-2


def _rel(a, b):
    a = a.double().cpu()
    b = b.double().cpu()
    return float((a - b).norm() / b.norm())


def test_noalloc_matches_handle_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    lib = dm.load()
    stream = torch.cuda.current_stream()
    gen = torch.Generator().manual_seed(2024)
    with dm.Handle(0) as h:
        for shape, sync in (((700, 300), 1), ((256, 1000), 0)):
            x = torch.randn(shape, generator=gen).cuda()
            ref = torch.empty_like(x)
            h.newton_schulz([x], [ref])
            out = torch.full_like(x, float("nan"))
            rc = lib.dmuon_newton_schulz_noalloc(
                ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(out.data_ptr()), shape[0], shape[1],
                5, None, 1e-7, sync, ctypes.c_void_p(stream.cuda_stream))
            assert rc == 0, dm.dmuon_error_string(rc)
            torch.cuda.synchronize()
            assert bool(torch.isfinite(out).all())
            e = _rel(out, ref)
            assert e <= NS_TOL, (shape, e)


def test_noalloc_rejects_sizes_beyond_its_limit():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    for shape in ((1025, 2048), (1024, 2049)):   # short side > 1024; rows*cols > 2^21
        x = torch.zeros(shape, device="cuda")
        o = torch.zeros(shape, device="cuda")
        rc = dm.dmuon_newton_schulz_noalloc(x.data_ptr(), o.data_ptr(), shape[0], shape[1])
        assert rc == -1
        assert float(o.abs().max()) == 0.0
    x = torch.zeros((8, 8), device="cuda")
    assert dm.dmuon_newton_schulz_noalloc(x.data_ptr() + 4, x.data_ptr(), 1, 1) == -2
    assert dm.dmuon_newton_schulz_noalloc(x.data_ptr(), x.data_ptr(), 8, 8) == -1

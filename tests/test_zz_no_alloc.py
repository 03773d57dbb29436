"""Allocation-free Newton-Schulz entry point (collected last on purpose).

dmuon_newton_schulz_noalloc serves callers that may not call cudaMalloc: a
host framework that owns all device memory, a plugin handed only its input
and output buffers, or a path that cannot take cudaMalloc's implicit
synchronisation.  Its scratch is a static device array shared by all calls.

These tests call it through the C ABI and compare its output with the fp64
oracle (relative Frobenius error 3e-2, the parity bar of every other GPU
test) and with the handle-based dmuon_newton_schulz: two calls in a row on
different shapes (so that a leftover of the first call would show in the
second), shapes at each of its documented limits, zero steps, a caller
table, a non-finite input in synchronous mode, and its refusal while the
stream is being captured.  They must pass alone in a fresh process and after
the rest of the suite.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import newton_schulz_nesterov_gb300 as dm  # noqa: E402
from newton_schulz_nesterov_gb300 import _build  # noqa: E402
import oracle  # noqa: E402

pytestmark = pytest.mark.gpu

NS_TOL = 3e-2


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _noalloc(x, out, ns_steps=5, coeffs=None, sync=1):
    stream = torch.cuda.current_stream()
    return dm.dmuon_newton_schulz_noalloc(x.data_ptr(), out.data_ptr(), x.shape[0], x.shape[1], ns_steps, coeffs,
                                          1e-7, bool(sync), stream)


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    return dm.load()


def test_noalloc_two_calls_match_oracle_and_handle_entry_point(lib):
    gen = torch.Generator().manual_seed(2024)
    with dm.Handle(0) as h:
        for shape, sync in (((700, 300), 1), ((256, 1000), 0)):
            x = torch.randn(shape, generator=gen)
            xd = x.cuda()
            ref_gpu = torch.empty_like(xd)
            h.newton_schulz([xd], [ref_gpu])
            out = torch.full_like(xd, float("nan"))
            stream = torch.cuda.current_stream()
            rc = lib.dmuon_newton_schulz_noalloc(
                ctypes.c_void_p(xd.data_ptr()), ctypes.c_void_p(out.data_ptr()), shape[0], shape[1],
                5, None, ctypes.c_float(1e-7), sync, ctypes.c_void_p(stream.cuda_stream))
            assert rc == 0, dm.dmuon_error_string(rc)
            torch.cuda.synchronize()
            assert bool(torch.isfinite(out).all())
            ref = oracle.newton_schulz(x.numpy().astype(np.float64))
            assert _rel(out.cpu().numpy(), ref) <= NS_TOL, shape
            assert _rel(out.cpu().numpy(), ref_gpu.cpu().numpy()) <= NS_TOL, shape


@pytest.mark.parametrize("shape", [(1024, 2048), (2048, 1024), (1, 1 << 21), (1 << 21, 1), (7, 299593)])
def test_noalloc_at_its_limits(lib, shape):
    """Short side exactly 1024 (both orientations), rows * cols exactly 2^21
    with one row or one column, and an odd short side whose padded rows
    reach the iterate buffer's slack, against the oracle."""
    x = torch.randn(shape, generator=torch.Generator().manual_seed(7))
    xd = x.cuda()
    out = torch.full_like(xd, float("nan"))
    assert _noalloc(xd, out) == 0
    ref = oracle.newton_schulz(x.numpy().astype(np.float64))
    assert _rel(out.cpu().numpy(), ref) <= NS_TOL, shape


def test_noalloc_zero_steps_and_caller_table(lib):
    x = torch.randn((300, 500), generator=torch.Generator().manual_seed(8))
    xd = x.cuda()
    out = torch.empty_like(xd)
    assert _noalloc(xd, out, ns_steps=0) == 0
    ref = x.numpy().astype(np.float64) / (np.linalg.norm(x.numpy().astype(np.float64)) + 1e-7)
    assert _rel(out.cpu().numpy(), ref) <= 1e-3   # the normalised input, rounded once to fp16
    table = [(3.0, -3.2, 1.2), (2.5, -2.0, 0.5), (1.875, -1.25, 0.375)]
    assert _noalloc(xd, out, ns_steps=3, coeffs=table) == 0
    assert _rel(out.cpu().numpy(), oracle.newton_schulz(x.numpy().astype(np.float64), 3, coeffs=table)) <= NS_TOL
    # a table that could leave fp16's range is refused before anything runs
    out.fill_(5.0)
    assert _noalloc(xd, out, ns_steps=3, coeffs=[(1.0, 25.0, 0.0)] * 3) == -1
    assert float(out.min()) == 5.0 and float(out.max()) == 5.0


def test_noalloc_nonfinite_input_in_sync_mode(lib):
    x = torch.randn((200, 300), device="cuda")
    x[3, 4] = float("nan")
    out = torch.empty_like(x)
    assert _noalloc(x, out, sync=1) == -5
    # the next call on a finite input starts clean
    y = torch.randn((200, 300), generator=torch.Generator().manual_seed(9))
    yd = y.cuda()
    assert _noalloc(yd, out, sync=1) == 0
    assert _rel(out.cpu().numpy(), oracle.newton_schulz(y.numpy().astype(np.float64))) <= NS_TOL


def test_noalloc_refuses_stream_capture(lib):
    """Each call uploads its descriptor from host memory, which a CUDA graph
    could not replay: under capture the call returns DMUON_ERR_ARG before any
    other CUDA call, and the output is untouched."""
    x = torch.randn((128, 256), device="cuda")
    out = torch.full_like(x, 7.0)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    rc = None
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            rc = dm.dmuon_newton_schulz_noalloc(x.data_ptr(), out.data_ptr(), 128, 256, 5, None, 1e-7, False, s)
    torch.cuda.synchronize()
    assert rc == -1
    assert float(out.min()) == 7.0 and float(out.max()) == 7.0


def test_noalloc_rejects_sizes_beyond_its_limit(lib):
    for shape in ((1025, 2048), (1024, 2049)):   # short side > 1024; rows*cols > 2^21
        x = torch.zeros(shape, device="cuda")
        o = torch.zeros(shape, device="cuda")
        rc = dm.dmuon_newton_schulz_noalloc(x.data_ptr(), o.data_ptr(), shape[0], shape[1])
        assert rc == -1
        assert float(o.abs().max()) == 0.0
    x = torch.zeros((8, 8), device="cuda")
    assert dm.dmuon_newton_schulz_noalloc(x.data_ptr() + 4, x.data_ptr(), 1, 1) == -2
    assert dm.dmuon_newton_schulz_noalloc(x.data_ptr(), x.data_ptr(), 8, 8) == -1

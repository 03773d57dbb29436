"""Python binding of libdmuon.so, the GB300 (sm_103a) owner-side Muon step.

Argument marshalling only: every step of the Muon update runs in the
library's CUDA kernels.  The functions keep the C names of
``include/dmuon.h``; PyTorch tensors are accepted for convenience (their
device pointers and shapes are passed through), raw device pointers with
explicit shapes are accepted by the ``*_ptrs`` variants.

There is no CPU fallback: if ``lib/libdmuon.so`` has not been built,
``load()`` raises.
"""
import ctypes
import os

__all__ = [
    "DmuonError", "load", "lib_path", "dmuon_create", "dmuon_destroy",
    "dmuon_step", "dmuon_step_ptrs", "dmuon_newton_schulz",
    "dmuon_newton_schulz_ptrs", "dmuon_newton_schulz_noalloc", "dmuon_get_status",
    "dmuon_gram_newton_schulz", "dmuon_gram_newton_schulz_ptrs", "BACKENDS",
    "dmuon_adamw_step", "dmuon_adamw_step_ptrs", "dmuon_clip_grad_norm", "dmuon_clip_grad_norm_ptrs",
    "dmuon_workspace_bytes", "dmuon_polar_express_coefficients", "dmuon_gram_check_coefficients",
    "dmuon_plan_preview",
    "dmuon_launch_count", "dmuon_last_error", "dmuon_profile_enable", "dmuon_profile_read",
    "dmuon_plan_summary", "dmuon_error_string", "dmuon_version", "Handle",
    "KIND_NAMES", "STATUS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "lib", "libdmuon.so")
_lib = None

STATUS = {
    0: "DMUON_OK", -1: "DMUON_ERR_ARG", -2: "DMUON_ERR_ALIGN", -3: "DMUON_ERR_OOM",
    -4: "DMUON_ERR_CUDA", -5: "DMUON_ERR_NONFINITE", -6: "DMUON_ERR_TIMEOUT",
    -7: "DMUON_ERR_UNSUPPORTED",
}
KIND_NAMES = ("momentum", "finalize", "gram", "gram2", "apply", "update0", "adamw", "clip", "small",
              "gs_gram", "gs_prod", "ns_fused")


class DmuonError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        msg = "%s (%d)" % (STATUS.get(code, "unknown"), code)
        if _lib is not None:
            msg += ": " + _lib.dmuon_error_string(code).decode()
        super().__init__(what + ": " + msg if what else msg)


class Shape(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


class Opts(ctypes.Structure):
    _fields_ = [("weight_decay", ctypes.c_float), ("eps", ctypes.c_float),
                ("nesterov", ctypes.c_int), ("scale_mode", ctypes.c_int),
                ("coeffs", ctypes.POINTER(ctypes.c_float)), ("backend", ctypes.c_int),
                ("restarts", ctypes.POINTER(ctypes.c_int)), ("n_restarts", ctypes.c_int)]


BACKENDS = {"direct": 0, "gram": 1}


def lib_path():
    return _LIB_PATH


def load(path=None):
    """Load libdmuon.so (once) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise ImportError("libdmuon.so not built (%s); run __graft_entry__.build()" % p)
    L = ctypes.CDLL(p)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    pp = ctypes.POINTER(ctypes.c_void_p)
    L.dmuon_default_opts.argtypes = [ctypes.POINTER(Opts)]
    L.dmuon_default_opts.restype = None
    L.dmuon_create.argtypes = [ctypes.POINTER(vp), i32]
    L.dmuon_create.restype = i32
    L.dmuon_destroy.argtypes = [vp]
    L.dmuon_destroy.restype = None
    L.dmuon_workspace_bytes.argtypes = [ctypes.POINTER(Shape), i32, ctypes.POINTER(ctypes.c_size_t)]
    L.dmuon_workspace_bytes.restype = i32
    L.dmuon_workspace_bytes_ex.argtypes = [ctypes.POINTER(Shape), i32, i32, ctypes.POINTER(ctypes.c_size_t)]
    L.dmuon_workspace_bytes_ex.restype = i32
    L.dmuon_gram_newton_schulz.argtypes = [vp, pp, pp, ctypes.POINTER(Shape), i32, i32,
                                           ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int),
                                           i32, f32, vp]
    L.dmuon_gram_newton_schulz.restype = i32
    L.dmuon_step.argtypes = [vp, pp, pp, pp, ctypes.POINTER(Shape), i32, f32, f32, i32,
                             ctypes.POINTER(Opts), vp]
    L.dmuon_step.restype = i32
    L.dmuon_newton_schulz.argtypes = [vp, pp, pp, ctypes.POINTER(Shape), i32, i32,
                                      ctypes.POINTER(ctypes.c_float), f32, vp]
    L.dmuon_newton_schulz.restype = i32
    L.dmuon_newton_schulz_noalloc.argtypes = [vp, vp, i64, i64, i32, ctypes.POINTER(ctypes.c_float),
                                              f32, i32, vp]
    L.dmuon_newton_schulz_noalloc.restype = i32
    L.dmuon_adamw_step.argtypes = [vp, pp, pp, pp, pp, ctypes.POINTER(i64), i32, f32, f32, f32, f32,
                                   f32, i32, vp]
    L.dmuon_adamw_step.restype = i32
    L.dmuon_clip_grad_norm.argtypes = [vp, pp, ctypes.POINTER(i64), i32, ctypes.POINTER(ctypes.c_int), i32,
                                       f32, ctypes.POINTER(f32), ctypes.POINTER(f32), vp]
    L.dmuon_clip_grad_norm.restype = i32
    L.dmuon_get_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int), i32]
    L.dmuon_get_status.restype = i32
    L.dmuon_last_error.argtypes = [vp]
    L.dmuon_last_error.restype = ctypes.c_char_p
    L.dmuon_set_overlap.argtypes = [vp, i32]
    L.dmuon_set_overlap.restype = i32
    L.dmuon_set_balanced_dealing.argtypes = [vp, i32]
    L.dmuon_set_balanced_dealing.restype = i32
    L.dmuon_set_fused_phases.argtypes = [vp, i32]
    L.dmuon_set_fused_phases.restype = i32
    L.dmuon_set_fp16_iterations.argtypes = [vp, i32]
    L.dmuon_set_fp16_iterations.restype = i32
    L.dmuon_set_small_path.argtypes = [vp, i32]
    L.dmuon_set_small_path.restype = i32
    L.dmuon_set_chunk_elements.argtypes = [vp, i64]
    L.dmuon_set_chunk_elements.restype = i32
    L.dmuon_set_tile_mode.argtypes = [vp, i32]
    L.dmuon_set_tile_mode.restype = i32
    L.dmuon_set_wait_timeout.argtypes = [vp, ctypes.c_uint64]
    L.dmuon_set_wait_timeout.restype = i32
    L.dmuon_launch_count.argtypes = [vp]
    L.dmuon_launch_count.restype = i64
    L.dmuon_profile_enable.argtypes = [vp, i32]
    L.dmuon_profile_enable.restype = i32
    L.dmuon_profile_read.argtypes = [vp, ctypes.POINTER(ctypes.c_double),
                                     ctypes.POINTER(ctypes.c_int64), i32]
    L.dmuon_profile_read.restype = i32
    L.dmuon_plan_summary.argtypes = [vp, ctypes.c_char_p, ctypes.c_size_t]
    L.dmuon_plan_summary.restype = i32
    L.dmuon_error_string.argtypes = [i32]
    L.dmuon_error_string.restype = ctypes.c_char_p
    L.dmuon_version.argtypes = []
    L.dmuon_version.restype = ctypes.c_char_p
    L.dmuon_plan_preview.argtypes = [ctypes.POINTER(Shape), i32, i32, i32, i32, i32, i32, ctypes.c_char_p,
                                     ctypes.c_size_t]
    L.dmuon_plan_preview.restype = i32
    L.dmuon_polar_express_coefficients.argtypes = [i32, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                                   ctypes.POINTER(ctypes.c_float)]
    L.dmuon_polar_express_coefficients.restype = i32
    L.dmuon_gram_check_coefficients.argtypes = [i32, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int),
                                                i32, ctypes.c_char_p, ctypes.c_size_t]
    L.dmuon_gram_check_coefficients.restype = i32
    _lib = L
    return L


def _check(code, what, h=None):
    if code != 0:
        if h is not None and _lib is not None:
            what = what + " [" + _lib.dmuon_last_error(h).decode() + "]"
        raise DmuonError(code, what)


def _ptr_array(ptrs):
    arr = (ctypes.c_void_p * max(1, len(ptrs)))()
    for i, p in enumerate(ptrs):
        arr[i] = int(p)
    return arr


def _shape_array(shapes):
    arr = (Shape * max(1, len(shapes)))()
    for i, (r, c) in enumerate(shapes):
        arr[i].rows, arr[i].cols = int(r), int(c)
    return arr


def _coeff_array(coeffs):
    if coeffs is None:
        return None
    flat = [float(v) for row in coeffs for v in row]
    return (ctypes.c_float * max(1, len(flat)))(*flat)


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def _tensor_args(tensors, name):
    ptrs, shapes = [], []
    for t in tensors:
        if t.dim() != 2 or not t.is_cuda or not t.is_contiguous() or str(t.dtype) != "torch.float32":
            raise ValueError("%s: each matrix must be a contiguous 2-D float32 CUDA tensor" % name)
        ptrs.append(t.data_ptr())
        shapes.append(tuple(t.shape))
    return ptrs, shapes


# ---------------------------------------------------------------- C calls

def dmuon_version():
    return load().dmuon_version().decode()


def dmuon_error_string(code):
    return load().dmuon_error_string(int(code)).decode()


def dmuon_create(device=0):
    h = ctypes.c_void_p()
    _check(load().dmuon_create(ctypes.byref(h), int(device)), "dmuon_create")
    return h


def dmuon_destroy(h):
    if h is not None:
        load().dmuon_destroy(h)


def dmuon_workspace_bytes(shapes, backend="direct"):
    out = ctypes.c_size_t(0)
    _check(load().dmuon_workspace_bytes_ex(_shape_array(shapes), len(shapes), BACKENDS[backend],
                                           ctypes.byref(out)), "dmuon_workspace_bytes")
    return out.value


def dmuon_polar_express_coefficients(steps=5, lower=1e-3, upper=1.0, safety=1.05):
    """Polar Express table (host only): ``steps`` rows (a, b, c) as floats."""
    out = (ctypes.c_float * (3 * max(1, int(steps))))()
    _check(load().dmuon_polar_express_coefficients(int(steps), float(lower), float(upper), float(safety), out),
           "dmuon_polar_express_coefficients")
    return [(out[3 * k], out[3 * k + 1], out[3 * k + 2]) for k in range(int(steps))]


def dmuon_plan_preview(shapes, backend="direct", tile_mode=0, clusters=76, sms=152, balanced=True):
    """Host-only summary of the plan a handle would build for ``shapes`` on a
    device with ``clusters`` 2-CTA clusters and ``sms`` SMs (GB300: 76, 152)."""
    buf = ctypes.create_string_buffer(512)
    rc = load().dmuon_plan_preview(_shape_array(shapes), len(shapes), BACKENDS[backend], int(tile_mode),
                                   int(clusters), int(sms), 1 if balanced else 0, buf, 512)
    if rc < 0:
        raise DmuonError(rc, "dmuon_plan_preview")
    return buf.value.decode()


def dmuon_gram_check_coefficients(ns_steps=5, coeffs=None, restarts=None):
    """The Gram-space backend's fp16 range check (host only): (True, "") or
    (False, reason)."""
    carr = _coeff_array(coeffs)
    rarr, nr = _restart_array(restarts)
    why = ctypes.create_string_buffer(256)
    rc = load().dmuon_gram_check_coefficients(int(ns_steps), carr, rarr, nr, why, 256)
    if rc not in (0, -1):
        raise DmuonError(rc, "dmuon_gram_check_coefficients")
    return rc == 0, why.value.decode()


def _restart_array(restarts):
    """None -> NULL (the default {2}); a sequence -> (int array, count)."""
    if restarts is None:
        return None, 0
    rs = [int(k) for k in restarts]
    return (ctypes.c_int * max(1, len(rs)))(*rs), len(rs)


def dmuon_step_ptrs(h, w_ptrs, g_ptrs, m_ptrs, shapes, lr, mu, ns_steps=5,
                    weight_decay=0.0, eps=1e-7, nesterov=True, scale_mode=0,
                    coeffs=None, stream=None, check=True, backend="direct", restarts=None):
    """dmuon_step on raw device pointers; returns the status code.
    backend "gram" selects the Gram-space iteration with restart positions
    `restarts` (None = the default [2])."""
    L = load()
    opts = Opts()
    L.dmuon_default_opts(ctypes.byref(opts))
    opts.weight_decay = float(weight_decay)
    opts.eps = float(eps)
    opts.nesterov = 1 if nesterov else 0
    opts.scale_mode = int(scale_mode)
    opts.backend = BACKENDS[backend]
    rarr, nr = _restart_array(restarts)
    if rarr is not None:
        opts.restarts = ctypes.cast(rarr, ctypes.POINTER(ctypes.c_int))
        opts.n_restarts = nr
    carr = _coeff_array(coeffs)
    if carr is not None:
        opts.coeffs = ctypes.cast(carr, ctypes.POINTER(ctypes.c_float))
    rc = L.dmuon_step(h, _ptr_array(w_ptrs), _ptr_array(g_ptrs), _ptr_array(m_ptrs),
                      _shape_array(shapes), len(shapes), float(lr), float(mu), int(ns_steps),
                      ctypes.byref(opts), ctypes.c_void_p(_stream_handle(stream)))
    if check:
        _check(rc, "dmuon_step", h)
    return rc


def dmuon_step(h, params, grads, momentum, lr=0.02, mu=0.95, ns_steps=5, **kw):
    """One Muon step over lists of CUDA fp32 tensors (updated in place)."""
    wp, ws = _tensor_args(params, "params")
    gp, gs = _tensor_args(grads, "grads")
    mp, ms = _tensor_args(momentum, "momentum")
    if ws != gs or ws != ms:
        raise ValueError("params, grads and momentum must have matching shapes")
    return dmuon_step_ptrs(h, wp, gp, mp, ws, lr, mu, ns_steps, **kw)


def dmuon_newton_schulz_ptrs(h, in_ptrs, out_ptrs, shapes, ns_steps=5, coeffs=None,
                             eps=1e-7, stream=None, check=True):
    L = load()
    carr = _coeff_array(coeffs)
    rc = L.dmuon_newton_schulz(h, _ptr_array(in_ptrs), _ptr_array(out_ptrs), _shape_array(shapes),
                               len(shapes), int(ns_steps),
                               None if carr is None else ctypes.cast(carr, ctypes.POINTER(ctypes.c_float)),
                               float(eps), ctypes.c_void_p(_stream_handle(stream)))
    if check:
        _check(rc, "dmuon_newton_schulz", h)
    return rc


def dmuon_newton_schulz(h, inputs, outputs, ns_steps=5, coeffs=None, eps=1e-7, stream=None):
    ip, is_ = _tensor_args(inputs, "inputs")
    op, os_ = _tensor_args(outputs, "outputs")
    if is_ != os_:
        raise ValueError("inputs and outputs must have matching shapes")
    return dmuon_newton_schulz_ptrs(h, ip, op, is_, ns_steps, coeffs, eps, stream)


def dmuon_gram_newton_schulz_ptrs(h, in_ptrs, out_ptrs, shapes, ns_steps=5, coeffs=None, restarts=None,
                                  eps=1e-7, stream=None, check=True):
    L = load()
    carr = _coeff_array(coeffs)
    rarr, nr = _restart_array(restarts)
    rc = L.dmuon_gram_newton_schulz(
        h, _ptr_array(in_ptrs), _ptr_array(out_ptrs), _shape_array(shapes), len(shapes), int(ns_steps),
        None if carr is None else ctypes.cast(carr, ctypes.POINTER(ctypes.c_float)),
        None if rarr is None else ctypes.cast(rarr, ctypes.POINTER(ctypes.c_int)), nr, float(eps),
        ctypes.c_void_p(_stream_handle(stream)))
    if check:
        _check(rc, "dmuon_gram_newton_schulz", h)
    return rc


def dmuon_gram_newton_schulz(h, inputs, outputs, ns_steps=5, coeffs=None, restarts=None, eps=1e-7,
                             stream=None):
    """Standalone Newton-Schulz with the Gram-space backend."""
    ip, is_ = _tensor_args(inputs, "inputs")
    op, os_ = _tensor_args(outputs, "outputs")
    if is_ != os_:
        raise ValueError("inputs and outputs must have matching shapes")
    return dmuon_gram_newton_schulz_ptrs(h, ip, op, is_, ns_steps, coeffs, restarts, eps, stream)


def dmuon_newton_schulz_noalloc(input_ptr, output_ptr, rows, cols, ns_steps=5, coeffs=None,
                                eps=1e-7, sync_status=True, stream=None):
    """Allocation-free standalone NS of one matrix (raw device pointers);
    returns the status code."""
    carr = _coeff_array(coeffs)
    return load().dmuon_newton_schulz_noalloc(
        ctypes.c_void_p(int(input_ptr)), ctypes.c_void_p(int(output_ptr)), int(rows), int(cols),
        int(ns_steps), None if carr is None else ctypes.cast(carr, ctypes.POINTER(ctypes.c_float)),
        float(eps), 1 if sync_status else 0, ctypes.c_void_p(_stream_handle(stream)))


def _flat_args(tensors, name):
    ptrs, numels = [], []
    for t in tensors:
        if not t.is_cuda or not t.is_contiguous() or str(t.dtype) != "torch.float32":
            raise ValueError("%s: each tensor must be a contiguous float32 CUDA tensor" % name)
        ptrs.append(t.data_ptr())
        numels.append(t.numel())
    return ptrs, numels


def dmuon_adamw_step_ptrs(h, p_ptrs, g_ptrs, m_ptrs, v_ptrs, numels, lr=1e-3, beta1=0.9,
                          beta2=0.999, eps=1e-8, weight_decay=0.01, step=1, stream=None, check=True):
    n = len(numels)
    nums = (ctypes.c_int64 * max(1, n))(*[int(x) for x in numels])
    rc = load().dmuon_adamw_step(h, _ptr_array(p_ptrs), _ptr_array(g_ptrs), _ptr_array(m_ptrs),
                                 _ptr_array(v_ptrs), nums, n, float(lr), float(beta1), float(beta2),
                                 float(eps), float(weight_decay), int(step),
                                 ctypes.c_void_p(_stream_handle(stream)))
    if check:
        _check(rc, "dmuon_adamw_step", h)
    return rc


def dmuon_adamw_step(h, params, grads, exp_avg, exp_avg_sq, **kw):
    """AdamW over lists of contiguous fp32 CUDA tensors (updated in place)."""
    pp_, nums = _flat_args(params, "params")
    gp, gn = _flat_args(grads, "grads")
    mp, mn = _flat_args(exp_avg, "exp_avg")
    vp_, vn = _flat_args(exp_avg_sq, "exp_avg_sq")
    if not (nums == gn == mn == vn):
        raise ValueError("params, grads, exp_avg, exp_avg_sq must have matching sizes")
    return dmuon_adamw_step_ptrs(h, pp_, gp, mp, vp_, nums, **kw)


def dmuon_clip_grad_norm_ptrs(h, g_ptrs, numels, max_norm, buckets=None, n_buckets=None,
                              stats=True, stream=None, check=True):
    """Returns (status, norms, coefs); norms/coefs are None when stats=False."""
    n = len(numels)
    nb = 1 if buckets is None else int(n_buckets if n_buckets is not None else max(buckets) + 1)
    nums = (ctypes.c_int64 * max(1, n))(*[int(x) for x in numels])
    bk = None if buckets is None else (ctypes.c_int * max(1, n))(*[int(b) for b in buckets])
    norms = (ctypes.c_float * nb)() if stats else None
    coefs = (ctypes.c_float * nb)() if stats else None
    rc = load().dmuon_clip_grad_norm(h, _ptr_array(g_ptrs), nums, n, bk, nb, float(max_norm),
                                     norms, coefs, ctypes.c_void_p(_stream_handle(stream)))
    if check:
        _check(rc, "dmuon_clip_grad_norm", h)
    if not stats:
        return rc, None, None
    return rc, [norms[i] for i in range(nb)], [coefs[i] for i in range(nb)]


def dmuon_clip_grad_norm(h, grads, max_norm, buckets=None, n_buckets=None, stats=True, stream=None):
    """Segmented clipping of CUDA fp32 gradients in place; returns (norms, coefs)."""
    gp, nums = _flat_args(grads, "grads")
    _, norms, coefs = dmuon_clip_grad_norm_ptrs(h, gp, nums, max_norm, buckets, n_buckets, stats, stream)
    return norms, coefs


def dmuon_get_status(h, n_flags=0):
    """Synchronise and return (status_code, per-matrix flags list)."""
    flags = (ctypes.c_int * max(1, n_flags))()
    rc = load().dmuon_get_status(h, flags, int(n_flags))
    return rc, [flags[i] for i in range(n_flags)]


def dmuon_set_overlap(h, on=True):  # default off in the library
    """Overlap the next chunk's momentum pass with the current chunk's products."""
    _check(load().dmuon_set_overlap(h, 1 if on else 0), "dmuon_set_overlap")


def dmuon_set_chunk_elements(h, elems):
    """Chunk size of later plans in matrix elements (0 = default 2^29)."""
    _check(load().dmuon_set_chunk_elements(h, int(elems)), "dmuon_set_chunk_elements")


def dmuon_set_balanced_dealing(h, on=True):  # default on in the library
    """Longest-first dealing of work items to the least-loaded CTA (pair) for later plans."""
    _check(load().dmuon_set_balanced_dealing(h, 1 if on else 0), "dmuon_set_balanced_dealing")


def dmuon_set_fp16_iterations(h, iters=3):  # default 3 in the library
    """Direct backend: leading Newton-Schulz iterations with fp16 operands
    (later ones bf16); 64 or more: every iteration."""
    _check(load().dmuon_set_fp16_iterations(h, int(iters)), "dmuon_set_fp16_iterations")


def dmuon_set_fused_phases(h, mode=2):  # default 2 (automatic) in the library
    """Direct backend: every product of every iteration of a chunk in one
    persistent launch -- 0 never, 1 always (True), 2 for chunks of few work
    items (the default); False selects 0."""
    m = 1 if mode is True else (0 if mode is False else int(mode))
    _check(load().dmuon_set_fused_phases(h, m), "dmuon_set_fused_phases")


def dmuon_set_small_path(h, on=True):  # default on in the library
    """Route small matrices (oriented m <= 128, n <= 512) through the fused
    one-CTA-per-matrix kernel (on) or through the chunked GEMM path (off)."""
    _check(load().dmuon_set_small_path(h, 1 if on else 0), "dmuon_set_small_path")


def dmuon_set_tile_mode(h, mode):
    """0 automatic, 1 single-CTA 128x256 tiles, 2 CTA-pair 256x256 tiles,
    3 single-CTA 128x128 tiles."""
    _check(load().dmuon_set_tile_mode(h, int(mode)), "dmuon_set_tile_mode")


def dmuon_set_wait_timeout(h, ns):
    _check(load().dmuon_set_wait_timeout(h, int(ns)), "dmuon_set_wait_timeout")


def dmuon_last_error(h):
    return load().dmuon_last_error(h).decode()


def dmuon_launch_count(h):
    return int(load().dmuon_launch_count(h))


def dmuon_profile_enable(h, on=True):
    _check(load().dmuon_profile_enable(h, 1 if on else 0), "dmuon_profile_enable")


def dmuon_profile_read(h):
    """{kind: (ms_total, launches)} accumulated since the last read."""
    n = len(KIND_NAMES)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    _check(load().dmuon_profile_read(h, ms, cnt, n), "dmuon_profile_read")
    return {KIND_NAMES[k]: (ms[k], cnt[k]) for k in range(n)}


def dmuon_plan_summary(h):
    L = load()
    need = L.dmuon_plan_summary(h, None, 0)
    buf = ctypes.create_string_buffer(need + 1)
    L.dmuon_plan_summary(h, buf, need + 1)
    return buf.value.decode()


class Handle:
    """Owning wrapper of a dmuon handle (destroyed on close / exit)."""

    def __init__(self, device=0):
        self.h = dmuon_create(device)

    def close(self):
        if self.h is not None:
            dmuon_destroy(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def step(self, params, grads, momentum, lr=0.02, mu=0.95, ns_steps=5, **kw):
        return dmuon_step(self.h, params, grads, momentum, lr, mu, ns_steps, **kw)

    def newton_schulz(self, inputs, outputs, ns_steps=5, coeffs=None, eps=1e-7, stream=None):
        return dmuon_newton_schulz(self.h, inputs, outputs, ns_steps, coeffs, eps, stream)

    def gram_newton_schulz(self, inputs, outputs, ns_steps=5, coeffs=None, restarts=None, eps=1e-7,
                           stream=None):
        return dmuon_gram_newton_schulz(self.h, inputs, outputs, ns_steps, coeffs, restarts, eps, stream)

    def status(self, n_flags=0):
        return dmuon_get_status(self.h, n_flags)

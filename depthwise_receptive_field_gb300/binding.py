"""ctypes binding of libwtconv's C ABI (include/wtconv.h and include/wtconv_ablation.h):
argument marshalling only.

Every function here has the name of the C entry point it calls and does no arithmetic of
its own. Tensor arguments may be torch tensors (their ``data_ptr()`` is passed), raw
integer device pointers, or None for optional arguments. ``stream`` may be a
``torch.cuda.Stream``, an integer handle, or None for torch's current stream.

The library is built from source on first use if it is missing or stale; if it cannot be
built or loaded, every call raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import build as _build

WT_OK, WT_ERR_INVALID_ARG, WT_ERR_UNSUPPORTED, WT_ERR_WORKSPACE, WT_ERR_CUDA, WT_ERR_TIMEOUT = range(6)
WT_F32, WT_BF16, WT_F16 = 0, 1, 2
(WT_VARIANT_REFERENCE, WT_VARIANT_FUSED_ANALYSIS, WT_VARIANT_COLLAPSED_SYNTHESIS,
 WT_VARIANT_FOLDED) = range(4)
VARIANT_NAMES = {WT_VARIANT_REFERENCE: "reference", WT_VARIANT_FUSED_ANALYSIS: "fused_analysis",
                 WT_VARIANT_COLLAPSED_SYNTHESIS: "collapsed_synthesis",
                 WT_VARIANT_FOLDED: "folded"}

HEADER = os.path.join(_build.INCLUDE, "wtconv.h")
HEADERS = [HEADER, os.path.join(_build.INCLUDE, "wtconv_ablation.h"),
           os.path.join(_build.INCLUDE, "wtconv_probe.h"),
           os.path.join(_build.INCLUDE, "wtconv_testing.h"),
           os.path.join(_build.INCLUDE, "wtconv_debug.h")]


class wt_desc(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int), ("c", ctypes.c_int), ("h", ctypes.c_int),
                ("w", ctypes.c_int), ("k", ctypes.c_int), ("levels", ctypes.c_int),
                ("io", ctypes.c_int)]

    def __repr__(self):
        return (f"wt_desc(n={self.n}, c={self.c}, h={self.h}, w={self.w}, k={self.k}, "
                f"levels={self.levels}, io={['f32', 'bf16', 'f16'][self.io]})")


class WTConvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


_LOCK = threading.Lock()
_LIB = None
_LIB_PATH = None  # None: the ordinary library (build.LIB)
_vp = ctypes.c_void_p
_DESC_P = ctypes.POINTER(wt_desc)

_SIGNATURES = {
    "wtconv_workspace_size": [_DESC_P, ctypes.POINTER(ctypes.c_size_t),
                              ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)],
    "wtconv_fold_scales": [_DESC_P] + [_vp] * 9,
    "wtconv_forward": [_DESC_P, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp],
    "wtconv_backward_data": [_DESC_P, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp],
    "wtconv_backward_weight": [_DESC_P] + [_vp] * 13 + [ctypes.c_size_t, _vp],
    "wtconv_backward": [_DESC_P] + [_vp] * 16 + [ctypes.c_size_t, _vp],
    "wtconv_backward_weight_noalloc": [_DESC_P] + [_vp] * 12 + [_vp],
    "wtconv_variant_workspace_size": [_DESC_P, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)],
    "wtconv_forward_variant": [_DESC_P, ctypes.c_int] + [_vp] * 8 + [ctypes.c_size_t, _vp],
    "wtconv_fma_probe": [ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp],
    "wtconv_workspace_status": [_vp, _vp, ctypes.POINTER(ctypes.c_int)],
    "wtconv_testing_set_wait_limit_ns": [ctypes.c_ulonglong],
    "wtconv_debug_phase_clocks": [ctypes.c_int, ctypes.c_int, _vp, ctypes.c_int],
}


def library_path() -> str:
    return _build.LIB


def use_library(path: str):
    """Load the calls from the library at `path` from now on (for the separately built
    phase-clock library, build.build_phase_clocks()); must precede the first call."""
    global _LIB_PATH
    with _LOCK:
        if _LIB is not None:
            raise RuntimeError("use_library must precede the first call into the library")
        _LIB_PATH = path


def load_library(rebuild_if_stale: bool = True):
    """Load (building first if needed) libwtconv.so and declare its signatures."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = _LIB_PATH or _build.LIB
            if _LIB_PATH is None and rebuild_if_stale and _build.stale():
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"libwtconv.so not found at {path}; run build() first")
            lib = ctypes.CDLL(path)
            for name, argtypes in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = argtypes
                fn.restype = ctypes.c_int
            lib.wtconv_status_string.argtypes = [ctypes.c_int]
            lib.wtconv_status_string.restype = ctypes.c_char_p
            lib.wtconv_last_launch_count.argtypes = []
            lib.wtconv_last_launch_count.restype = ctypes.c_int
            _LIB = lib
    return _LIB


def declared_functions() -> list[str]:
    """Names of the functions the public headers (include/*.h) declare."""
    names = set()
    for h in HEADERS:
        text = open(h).read()
        names.update(re.findall(r"^\s*(?:wt_status|const char\*|int)\s+(wtconv_\w+)\s*\(",
                                text, flags=re.M))
    return sorted(names)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _dev(t, what: str, dtype=None, numel=None):
    """Device pointer of a tensor argument, after the checks the C ABI cannot make from a
    raw pointer: contiguous, of the expected dtype and size, on a CUDA device. None and
    raw integer addresses pass through unchecked (the ABI's own tests of null and
    misaligned pointers use them)."""
    if t is None or isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError(f"{what}: the tensor must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what}: dtype {t.dtype}, expected {dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{what}: {t.numel()} elements, expected {numel}")
    if not t.is_cuda:
        raise ValueError(f"{what}: a CUDA tensor is required")
    return t.data_ptr()


def _io_dtype(desc):
    import torch
    return {WT_F32: torch.float32, WT_BF16: torch.bfloat16, WT_F16: torch.float16}[desc.io]


def _sizes(desc):
    """Element counts of a plane tensor and of the parameter arrays of desc."""
    kk, c, L = desc.k * desc.k, desc.c, desc.levels
    return {"x": desc.n * c * desc.h * desc.w, "w0": c * kk, "c": c, "wl": L * c * 4 * kk,
            "sl": L * c * 4}


def _ws(ws, ws_bytes, what: str):
    if ws is not None and not isinstance(ws, int) and \
            ws.numel() * ws.element_size() < int(ws_bytes):
        raise ValueError(f"{what}: workspace of {ws.numel() * ws.element_size()} bytes, "
                         f"ws_bytes says {int(ws_bytes)}")
    return _dev(ws, what + " (workspace)")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str):
    if status != WT_OK:
        raise WTConvError(status, where)


def status_string(status: int) -> str:
    return load_library().wtconv_status_string(int(status)).decode()


def make_desc(n, c, h, w, k, levels, io) -> wt_desc:
    if not isinstance(io, int):
        import torch
        io = {torch.bfloat16: WT_BF16, torch.float16: WT_F16}.get(io, WT_F32)
    return wt_desc(int(n), int(c), int(h), int(w), int(k), int(levels), int(io))


def desc_like(x, k: int, levels: int) -> wt_desc:
    n, c, h, w = x.shape
    return make_desc(n, c, h, w, k, levels, x.dtype)


def wtconv_workspace_size(desc: wt_desc):
    """Returns (fwd, bwd_data, bwd_weight) workspace bytes."""
    a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(load_library().wtconv_workspace_size(ctypes.byref(desc), ctypes.byref(a),
                                                ctypes.byref(b), ctypes.byref(c)),
           "wtconv_workspace_size")
    return a.value, b.value, c.value


def _params(desc, where, **named):
    """Device pointers of fp32 parameter-shaped arguments, by name: w0-like [C,k,k],
    c-like [C], wl-like [L,C,4,k,k], sl-like [L,C,4]."""
    import torch
    n = _sizes(desc)
    kind = {"w0": "w0", "w0f": "w0", "dw0": "w0", "b0": "c", "s0": "c", "b0f": "c",
            "db0": "c", "ds0": "c", "wl": "wl", "wlf": "wl", "dwl": "wl", "sl": "sl",
            "dsl": "sl"}
    return {k: _dev(v, f"{where}: {k}", torch.float32, n[kind[k]]) for k, v in named.items()}


def _plane(desc, where, name, t):
    return _dev(t, f"{where}: {name}", _io_dtype(desc), _sizes(desc)["x"])


def wtconv_fold_scales(desc, w0, b0, s0, wl, sl, w0f, b0f, wlf, stream=None):
    w = "wtconv_fold_scales"
    p = _params(desc, w, w0=w0, b0=b0, s0=s0, wl=wl, sl=sl, w0f=w0f, b0f=b0f, wlf=wlf)
    _check(load_library().wtconv_fold_scales(
        ctypes.byref(desc), p["w0"], p["b0"], p["s0"], p["wl"], p["sl"], p["w0f"], p["b0f"],
        p["wlf"], _stream(stream)), w)


def wtconv_forward(desc, x, w0f, b0f, wlf, y, ws=None, ws_bytes=0, stream=None):
    w = "wtconv_forward"
    p = _params(desc, w, w0f=w0f, b0f=b0f, wlf=wlf)
    _check(load_library().wtconv_forward(
        ctypes.byref(desc), _plane(desc, w, "x", x), p["w0f"], p["b0f"], p["wlf"],
        _plane(desc, w, "y", y), _ws(ws, ws_bytes, w), int(ws_bytes), _stream(stream)), w)


def wtconv_backward_data(desc, dy, w0f, wlf, dx, ws=None, ws_bytes=0, stream=None):
    w = "wtconv_backward_data"
    p = _params(desc, w, w0f=w0f, wlf=wlf)
    _check(load_library().wtconv_backward_data(
        ctypes.byref(desc), _plane(desc, w, "dy", dy), p["w0f"], p["wlf"],
        _plane(desc, w, "dx", dx), _ws(ws, ws_bytes, w), int(ws_bytes), _stream(stream)), w)


def wtconv_backward_weight(desc, x, dy, w0, b0, s0, wl, sl, dw0, db0, ds0, dwl, dsl, ws,
                           ws_bytes, stream=None):
    w = "wtconv_backward_weight"
    p = _params(desc, w, w0=w0, b0=b0, s0=s0, wl=wl, sl=sl, dw0=dw0, db0=db0, ds0=ds0,
                dwl=dwl, dsl=dsl)
    _check(load_library().wtconv_backward_weight(
        ctypes.byref(desc), _plane(desc, w, "x", x), _plane(desc, w, "dy", dy), p["w0"],
        p["b0"], p["s0"], p["wl"], p["sl"], p["dw0"], p["db0"], p["ds0"], p["dwl"], p["dsl"],
        _ws(ws, ws_bytes, w), int(ws_bytes), _stream(stream)), w)


def wtconv_backward(desc, x, dy, w0f, wlf, w0, b0, s0, wl, sl, dx, dw0, db0, ds0, dwl, dsl,
                    ws, ws_bytes, stream=None):
    w = "wtconv_backward"
    p = _params(desc, w, w0f=w0f, wlf=wlf, w0=w0, b0=b0, s0=s0, wl=wl, sl=sl, dw0=dw0,
                db0=db0, ds0=ds0, dwl=dwl, dsl=dsl)
    _check(load_library().wtconv_backward(
        ctypes.byref(desc), _plane(desc, w, "x", x), _plane(desc, w, "dy", dy), p["w0f"],
        p["wlf"], p["w0"], p["b0"], p["s0"], p["wl"], p["sl"], _plane(desc, w, "dx", dx),
        p["dw0"], p["db0"], p["ds0"], p["dwl"], p["dsl"], _ws(ws, ws_bytes, w), int(ws_bytes),
        _stream(stream)), w)


def wtconv_backward_weight_noalloc(desc, x, dy, w0, b0, s0, wl, sl, dw0, db0, ds0, dwl, dsl,
                                   stream=None):
    """Backward-weight with the library's built-in 4 MiB scratch (no workspace)."""
    w = "wtconv_backward_weight_noalloc"
    p = _params(desc, w, w0=w0, b0=b0, s0=s0, wl=wl, sl=sl, dw0=dw0, db0=db0, ds0=ds0,
                dwl=dwl, dsl=dsl)
    _check(load_library().wtconv_backward_weight_noalloc(
        ctypes.byref(desc), _plane(desc, w, "x", x), _plane(desc, w, "dy", dy), p["w0"],
        p["b0"], p["s0"], p["wl"], p["sl"], p["dw0"], p["db0"], p["ds0"], p["dwl"], p["dsl"],
        _stream(stream)), w)


def wtconv_variant_workspace_size(desc: wt_desc, variant: int) -> int:
    """Workspace bytes of wtconv_forward_variant for (desc, variant)."""
    n = ctypes.c_size_t()
    _check(load_library().wtconv_variant_workspace_size(ctypes.byref(desc), int(variant),
                                                        ctypes.byref(n)),
           "wtconv_variant_workspace_size")
    return n.value


def wtconv_forward_variant(desc, variant, x, w0, b0, s0, wl, sl, y, ws, ws_bytes, stream=None):
    _check(load_library().wtconv_forward_variant(
        ctypes.byref(desc), int(variant), _ptr(x), _ptr(w0), _ptr(b0), _ptr(s0), _ptr(wl),
        _ptr(sl), _ptr(y), _ptr(ws), int(ws_bytes), _stream(stream)), "wtconv_forward_variant")


def wtconv_workspace_status(ws, stream=None) -> int:
    """Bit flags of the calls whose kernels timed out on this workspace (0 = none); see
    include/wtconv.h. Synchronizes the stream."""
    flags = ctypes.c_int(0)
    st = load_library().wtconv_workspace_status(_ptr(ws), _stream(stream), ctypes.byref(flags))
    if st not in (WT_OK, WT_ERR_TIMEOUT):
        _check(st, "wtconv_workspace_status")
    return flags.value


def wtconv_testing_set_wait_limit_ns(ns: int):
    """Test hook (include/wtconv_testing.h): limit of the kernels' bounded waits; 0 = 1 s."""
    _check(load_library().wtconv_testing_set_wait_limit_ns(int(ns)),
           "wtconv_testing_set_wait_limit_ns")


def wtconv_debug_phase_clocks(kernel: int, reset: bool = False) -> list:
    """The 32 phase counters of a plane kernel (include/wtconv_debug.h): 0 forward /
    backward-data, 1 backward-weight. Raises WTConvError (WT_ERR_UNSUPPORTED) unless the
    library was built with the clocks."""
    buf = (ctypes.c_ulonglong * 32)()
    _check(load_library().wtconv_debug_phase_clocks(int(kernel), 1 if reset else 0,
                                                    ctypes.cast(buf, _vp), 32),
           "wtconv_debug_phase_clocks")
    return list(buf)


def wtconv_fma_probe(blocks: int, iters: int, packed: bool, out, stream=None):
    """Launch the FP32 multiply-add throughput probe (include/wtconv_probe.h)."""
    _check(load_library().wtconv_fma_probe(int(blocks), int(iters), 1 if packed else 0,
                                           _ptr(out), _stream(stream)), "wtconv_fma_probe")


def wtconv_status_string(status: int) -> str:
    return status_string(status)


def wtconv_last_launch_count() -> int:
    return int(load_library().wtconv_last_launch_count())

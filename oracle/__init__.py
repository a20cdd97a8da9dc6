"""CPU oracle for the WTConv layer: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg of
``bench.py`` may import this package. The CUDA product path never calls it, and the two
share no code: the oracle is plain C loops in double precision (``wtconv_oracle.c``),
compiled with gcc and loaded here with ctypes.

What it computes follows "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware
Reformulation" (Aflalo et al.):

* ``forward(..., mode="cascade")`` -- Algorithm 1 (§2.1) with every intermediate
  materialized and the level-by-level synthesis cascade;
* ``forward(..., mode="closed")`` -- the same filtered coefficients Z^(l) summed with the
  closed-form bit-indexed synthesis of Prop. 2 (Eq. 6-7);
* ``backward`` -- the literal reverse-mode derivative of Algorithm 1 with respect to the
  input and the unfolded parameters (W^(0), b, s^(0), W^(l), s^(l));
* ``haar_analysis`` / ``haar_synthesis`` / ``dwconv`` -- the building blocks (Eq. 5,
  Eq. 12, zero-padded depthwise cross-correlation), exposed for the pins.

Every function is pinned by ``tests/test_oracle_pins.py`` against something other than
itself (Prop. 1, Eq. 13, library convolutions with autograd, exact reconstruction,
finite differences, a brute-force operator matrix).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wtconv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libwtconv_oracle.so")
_LOCK = threading.Lock()
_LIB = None


class _Desc(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in ("n", "c", "h", "w", "k", "levels")]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, strict IEEE: no -ffast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = build()
            lib = ctypes.CDLL(path)
            dp = ctypes.POINTER(ctypes.c_double)
            lib.wo_forward.argtypes = [ctypes.POINTER(_Desc), dp, dp, dp, dp, dp, dp, dp,
                                       ctypes.c_int]
            lib.wo_forward.restype = ctypes.c_int
            lib.wo_backward.argtypes = [ctypes.POINTER(_Desc)] + [dp] * 13
            lib.wo_backward.restype = ctypes.c_int
            lib.wo_haar_analysis.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp]
            lib.wo_haar_synthesis.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp]
            lib.wo_dwconv.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp, dp]
            lib.wo_num_threads.restype = ctypes.c_int
            lib.wo_set_num_threads.argtypes = [ctypes.c_int]
            lib.wo_set_num_threads.restype = None
            _LIB = lib
    return _LIB


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def num_threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all cores)."""
    return int(_lib().wo_num_threads())


def set_num_threads(n: int) -> None:
    """OpenMP threads for the following calls (the timed CPU baseline's single-thread leg)."""
    _lib().wo_set_num_threads(int(n))


def _desc(x, k, levels):
    n, c, h, w = x.shape
    return _Desc(n, c, h, w, k, levels)


def forward(x, w0, b0, s0, wl, sl, levels: int, mode: str = "cascade") -> np.ndarray:
    """WTConv forward in float64. x [N,C,H,W]; w0 [C,k,k]; b0 [C] or None; s0 [C];
    wl [L,C,4,k,k]; sl [L,C,4]. mode "cascade" (Algorithm 1) or "closed" (Eq. 7)."""
    x, w0, b0, s0 = _f64(x), _f64(w0), _f64(b0), _f64(s0)
    k = w0.shape[-1]
    if levels > 0:
        wl, sl = _f64(wl), _f64(sl)
    else:
        wl = sl = None
    y = np.empty_like(x)
    rc = _lib().wo_forward(ctypes.byref(_desc(x, k, levels)), _ptr(x), _ptr(w0), _ptr(b0),
                           _ptr(s0), _ptr(wl), _ptr(sl), _ptr(y),
                           {"cascade": 0, "closed": 1}[mode])
    if rc != 0:
        raise ValueError(f"oracle forward failed with code {rc}")
    return y


def backward(x, dy, w0, b0, s0, wl, sl, levels: int) -> dict:
    """Literal reverse mode of Algorithm 1. Returns dx, dw0, db0, ds0, dwl, dsl (float64)."""
    x, dy, w0, b0, s0 = _f64(x), _f64(dy), _f64(w0), _f64(b0), _f64(s0)
    c, k = w0.shape[0], w0.shape[-1]
    if levels > 0:
        wl, sl = _f64(wl), _f64(sl)
    else:
        wl = sl = None
    out = {
        "dx": np.empty_like(x),
        "dw0": np.empty_like(w0),
        "db0": np.empty(c),
        "ds0": np.empty(c),
        "dwl": np.empty((max(levels, 0), c, 4, k, k)),
        "dsl": np.empty((max(levels, 0), c, 4)),
    }
    rc = _lib().wo_backward(
        ctypes.byref(_desc(x, k, levels)), _ptr(x), _ptr(dy), _ptr(w0), _ptr(b0), _ptr(s0),
        _ptr(wl), _ptr(sl), _ptr(out["dx"]), _ptr(out["dw0"]), _ptr(out["db0"]),
        _ptr(out["ds0"]), _ptr(out["dwl"]) if levels > 0 else None,
        _ptr(out["dsl"]) if levels > 0 else None)
    if rc != 0:
        raise ValueError(f"oracle backward failed with code {rc}")
    return out


def haar_analysis(img) -> np.ndarray:
    """Eq. 5 on every 2x2 block of one plane [h, w] -> [4, ceil(h/2), ceil(w/2)]
    (LL, LH, HL, HH); pixels past an odd edge are zero."""
    img = _f64(img)
    h, w = img.shape
    out = np.empty((4, (h + 1) // 2, (w + 1) // 2))
    _lib().wo_haar_analysis(h, w, _ptr(img), _ptr(out))
    return out


def haar_synthesis(bands) -> np.ndarray:
    """Eq. 12 on one level of coefficients [4, h2, w2] -> plane [2*h2, 2*w2]."""
    bands = _f64(bands)
    _, h2, w2 = bands.shape
    out = np.empty((2 * h2, 2 * w2))
    _lib().wo_haar_synthesis(h2, w2, _ptr(bands), _ptr(out))
    return out


def dwconv(img, wt) -> np.ndarray:
    """Zero-padded 'same' cross-correlation of one plane [h, w] with one kernel [k, k]."""
    img, wt = _f64(img), _f64(wt)
    h, w = img.shape
    out = np.empty_like(img)
    _lib().wo_dwconv(h, w, wt.shape[0], _ptr(img), _ptr(wt), _ptr(out))
    return out

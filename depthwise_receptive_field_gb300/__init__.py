"""GB300-native (sm_103a) WTConv layer: forward and backward of the wavelet convolution.

The computation lives in ``libwtconv.so`` (hand-written CUDA kernels behind the C ABI of
``include/wtconv.h``). ``binding`` is the thin ctypes layer with the C names, ``layer`` a
convenience wrapper that allocates with torch, ``inputs`` the seeded synthetic inputs,
``iomodel`` the paper's traffic/arithmetic models used for reporting.

Importing this package loads nothing; the library is loaded (and built if stale) on first
use, and every entry point raises if it cannot be loaded: there is no CPU fallback.
"""

__all__ = ["binding", "layer", "inputs", "iomodel", "build"]

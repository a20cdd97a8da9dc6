"""Build libwtconv.so (the CUDA kernels and the C ABI) for sm_103a, in-tree.

Each .cu translation unit is compiled in parallel with nvcc, then linked into one shared
library (CUDA runtime linked statically, so the library loads without a GPU).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libwtconv.so")
# the same library with the plane kernels' per-phase clocks compiled in (analysis only)
PHASE_BUILD = os.path.join(BUILD, "phase")
PHASE_LIB = os.path.join(PHASE_BUILD, "libwtconv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", f"-I{INCLUDE}"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libwtconv")
    return path


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]


def stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=None, out_dir: str = BUILD) -> str:
    """Compile and link into out_dir/libwtconv.so; returns the library path. Rebuilds only
    when sources changed."""
    lib_path = os.path.join(out_dir, "libwtconv.so")
    if not force and not stale(lib_path):
        return lib_path
    os.makedirs(out_dir, exist_ok=True)
    extra = list(extra_flags or [])
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src).replace(".cu", ".o"))
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        return obj, res.stderr

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, _sources()))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", *[o for o, _ in results], "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


def build_phase_clocks(force: bool = False) -> str:
    """The library with the plane kernels' per-phase clocks (-DWT_PHASE_CLOCKS), built apart
    from the ordinary one; returns its path."""
    return build(force=force, extra_flags=["-DWT_PHASE_CLOCKS"], out_dir=PHASE_BUILD)


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)

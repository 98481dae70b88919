"""Build the CUDA library ``libfp8rl.so`` in-tree for sm_103a.

Each ``csrc/*.cu`` is compiled to an object in parallel with one
``-gencode arch=compute_103a,code=sm_103a`` and linked into one shared library
next to this file.  The CUDA runtime is linked dynamically so that the library
shares the process's runtime (and its streams) with PyTorch.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfp8rl.so")
# debug flavour (FP8RL_DEBUG=1): device-side checks of every store index,
# failures reported as FP8RL_ERR_DEVICE_CHECK instead of a store
LIB_DEBUG = os.path.join(PKG, "libfp8rl_debug.so")
INCLUDE = os.path.join(ROOT, "include")


def debug_requested() -> bool:
    return os.environ.get("FP8RL_DEBUG") == "1"


def lib_path(debug: bool | None = None) -> str:
    """The library of the requested flavour (default: FP8RL_DEBUG=1 selects
    the debug build)."""
    return LIB_DEBUG if (debug_requested() if debug is None else debug) else LIB

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def cuda_home() -> str:
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return cand
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(nvcc))
    raise RuntimeError("nvcc not found (set CUDA_HOME)")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        [os.path.join(INCLUDE, "fp8rl.h"), os.path.abspath(__file__)]


def up_to_date(debug: bool = False) -> bool:
    lib = lib_path(debug)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, debug: bool | None = None) -> str:
    """Compile (if stale) and return the path of ``libfp8rl.so`` (or, for the
    debug flavour, ``libfp8rl_debug.so``)."""
    debug = debug_requested() if debug is None else debug
    lib = lib_path(debug)
    if not force and up_to_date(debug):
        return lib
    home = cuda_home()
    nvcc = os.path.join(home, "bin", "nvcc")
    build_dir = os.path.join(BUILD, "debug") if debug else BUILD
    os.makedirs(build_dir, exist_ok=True)
    procs = []
    objs = []
    for src in _sources():
        obj = os.path.join(build_dir, os.path.basename(src).replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *(["-DFP8RL_DEBUG"] if debug else []), "-I", INCLUDE, "-c", src, "-o", obj]
        if verbose:
            cmd += ["-Xptxas", "-v"]
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((src, text))
        elif verbose and text.strip():
            sys.stderr.write(f"== {os.path.basename(src)}\n{text}\n")
    if failed:
        msg = "\n".join(f"== {s}\n{t}" for s, t in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = lib + f".{os.getpid()}.tmp"
    link = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
            f"-L{home}/lib64", "-Xlinker", f"-rpath,{home}/lib64"]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug=True if "--debug" in sys.argv else None))

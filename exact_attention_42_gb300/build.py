"""Builds libfa.so (the C-ABI library) in-tree with nvcc for sm_103a."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG_DIR, "libfa.so")
# The same library compiled with FA_DEBUG: every computed TMA coordinate,
# output row and TMEM base column is checked before use (see include/fa.h).
DEBUG_LIB_PATH = os.path.join(PKG_DIR, "libfa_debug.so")
SOURCES = [os.path.join(CSRC, n)
           for n in ("fa_api.cu", "fa_fwd.cu", "fa_decode.cu", "fa_bwd.cu", "fa_quant.cu", "fa_sched.cu", "fa_host.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, "ptx.cuh"), os.path.join(CSRC, "fa_internal.h"), os.path.join(INCLUDE, "fa.h")]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"),
                 os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; set CUDA_HOME or NVCC")


def _stale(path: str) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(f) > t for f in DEPENDS)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compiles the library if a source is newer than it; returns its path.
    debug=True builds libfa_debug.so, with the FA_DEBUG checks compiled in."""
    path = DEBUG_LIB_PATH if debug else LIB_PATH
    if not force and not _stale(path):
        return path
    tmp = path + ".tmp.%d" % os.getpid()
    cmd = [nvcc_path(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "--threads", "0",
           "-I", INCLUDE, "-I", CSRC, *(["-DFA_DEBUG"] if debug else []), "-o", tmp, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n%s\n%s" % (" ".join(cmd), res.stderr))
    if verbose:
        print(res.stderr)
    os.replace(tmp, path)
    return path

"""In-tree build of the CUDA library (and of the test-only unit-kernel library).

    python -m exact_attention_68_gb300.build      # builds both, prints the paths

One nvcc invocation per shared object, sm_103a only, translation units
compiled in parallel.  A build is skipped when the .so is newer than every
source it is made from.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "lib")
LIB_PATH = os.path.join(LIBDIR, "libattn_sm103.so")
DEBUG_LIB_PATH = os.path.join(LIBDIR, "libattn_sm103_debug.so")
UNIT_SRC = os.path.join(ROOT, "tests", "cuda", "umma_unit.cu")
UNIT_LIB = os.path.join(ROOT, "tests", "cuda", "libumma_unit.so")
SCHED_SRC = os.path.join(ROOT, "tests", "cuda", "sched_check.cpp")
SCHED_LIB = os.path.join(ROOT, "tests", "cuda", "libsched_check.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-shared",
         "-Xcompiler", "-fvisibility=hidden", "--threads", "4",
         "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return [os.path.join(CSRC, f) for f in ("attn_api.cu", "attn_fwd_1q_sm103.cu", "attn_fwd_1qp_sm103.cu",
                                            "attn_noalloc.cu", "attn_bwd_api.cu", "attn_bwd_sm103.cu", "attn_bwd256_sm103.cu")]


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "attn.h"))
    return files


def _stale(target, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + r.stdout + r.stderr)
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)


def build_library(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Build libattn_sm103.so (the product library) in-tree; return its path."""
    os.makedirs(LIBDIR, exist_ok=True)
    if force or _stale(LIB_PATH, _deps()):
        tmp = LIB_PATH + ".tmp"
        _run([_nvcc(), *ARCH, *FLAGS, *extra, "-o", tmp, *_sources()], verbose)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def build_debug_library(force: bool = False, verbose: bool = False) -> str:
    """Build the debug variant of the library (-DATTN_DEBUG: every kernel checks
    its index arithmetic before each memory access and reports a failed check
    as ATTN_ERR_DEVICE_CHECK instead of making the access); return its path."""
    os.makedirs(LIBDIR, exist_ok=True)
    if force or _stale(DEBUG_LIB_PATH, _deps()):
        tmp = DEBUG_LIB_PATH + ".tmp"
        _run([_nvcc(), *ARCH, *FLAGS, "-DATTN_DEBUG", "-o", tmp, *_sources()], verbose)
        os.replace(tmp, DEBUG_LIB_PATH)
    return DEBUG_LIB_PATH


def build_unit_library(force: bool = False, verbose: bool = False) -> str:
    """Build the test-only tcgen05 descriptor unit kernels; return the path."""
    if force or _stale(UNIT_LIB, _deps() + [UNIT_SRC]):
        tmp = UNIT_LIB + ".tmp"
        _run([_nvcc(), *ARCH, *FLAGS, "-o", tmp, UNIT_SRC], verbose)
        os.replace(tmp, UNIT_LIB)
    return UNIT_LIB


def build_sched_check(force: bool = False, verbose: bool = False) -> str:
    """Build the test-only host shim over the grid schedule (g++, no CUDA)."""
    hdr = os.path.join(CSRC, "schedule.h")
    if force or _stale(SCHED_LIB, [hdr, SCHED_SRC]):
        tmp = SCHED_LIB + ".tmp"
        cxx = os.environ.get("CXX") or shutil.which("g++") or "g++"
        _run([cxx, "-O2", "-std=c++17", "-fPIC", "-shared", "-fvisibility=hidden",
              "-I", CSRC, "-o", tmp, SCHED_SRC], verbose)
        os.replace(tmp, SCHED_LIB)
    return SCHED_LIB


if __name__ == "__main__":
    force = "--force" in sys.argv
    print(build_library(force=force, verbose=True))
    print(build_unit_library(force=force, verbose=True))
    print(build_sched_check(force=force, verbose=True))

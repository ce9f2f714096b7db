"""Builds libfa.so (the CUDA kernels and their C ABI) in this directory.

One nvcc invocation per translation unit, run in parallel, for sm_103a only,
then one link step.  Objects go to ``_build/`` beside this file; the shared
library lands next to this file as ``libfa.so`` where the binding loads it.
"""
from __future__ import annotations

import os
import platform
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfa.so")
SOURCES = ["api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_decode.cu", "fa_fp8.cu", "page_pool.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", os.path.join(HERE, "..", "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa.so")


def _deps(src: str):
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] + [
        os.path.join(HERE, "..", "include", "fa.h"), src]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build(verbose: bool = False, force: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    stamp = os.path.join(BUILD, "host_arch")
    arch = platform.machine()
    if not os.path.exists(stamp) or open(stamp).read().strip() != arch:
        force = True  # objects built on another host architecture cannot be linked here
    with open(stamp, "w") as f:
        f.write(arch)
    jobs = []
    objs = []
    for name in SOURCES:
        src = os.path.join(CSRC, name)
        obj = os.path.join(BUILD, os.path.splitext(name)[0] + ".o")
        objs.append(obj)
        if force or _stale(obj, _deps(src)):
            jobs.append([nvcc, *ARCH, *FLAGS, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        if verbose:
            print(r.stdout + r.stderr)

    with ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(LIB, objs):
        run([nvcc, *ARCH, "-shared", "-o", LIB, *objs])
    return LIB


COUNT_LIB = os.path.join(HERE, "libfa_count.so")


def build_counting(verbose: bool = False) -> str:
    """A test-only variant of the library: the forward kernel compiled with
    FA_COUNT_RESCALES, which counts the lazy rescales it takes per (batch,
    head) and exports fa_test_rescale_counts().  Linked from the product's
    other objects; the product libfa.so never contains the counter."""
    build(verbose=verbose)
    obj = os.path.join(BUILD, "fa_fwd_count.o")
    src = os.path.join(CSRC, "fa_fwd.cu")
    nvcc = _nvcc()

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)

    if _stale(obj, _deps(src)):
        run([nvcc, *ARCH, *FLAGS, "-DFA_COUNT_RESCALES", "-c", src, "-o", obj])
    objs = [obj if n == "fa_fwd.cu" else os.path.join(BUILD, os.path.splitext(n)[0] + ".o") for n in SOURCES]
    if _stale(COUNT_LIB, objs):
        run([nvcc, *ARCH, "-shared", "-o", COUNT_LIB, *objs])
    return COUNT_LIB


BOUNDS_LIB = os.path.join(HERE, "libfa_bounds.so")
BOUNDS_SOURCES = ("fa_fwd.cu", "fa_bwd.cu", "fa_decode.cu")


def build_bounds(verbose: bool = False) -> str:
    """A test-only variant of the library: the forward, backward and decode
    kernels compiled with FA_BOUNDS_CHECK, so that every plain (non-TMA)
    global load, store and atomic they make checks its index against its
    buffer and records an error code instead of touching memory outside it.
    Linked from the product's other objects; the product libfa.so has no
    checks."""
    build(verbose=verbose)
    nvcc = _nvcc()

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)

    objs, jobs = [], []
    for n in SOURCES:
        if n in BOUNDS_SOURCES:
            src = os.path.join(CSRC, n)
            obj = os.path.join(BUILD, os.path.splitext(n)[0] + "_bounds.o")
            if _stale(obj, _deps(src)):
                jobs.append([nvcc, *ARCH, *FLAGS, "-DFA_BOUNDS_CHECK", "-c", src, "-o", obj])
            objs.append(obj)
        else:
            objs.append(os.path.join(BUILD, os.path.splitext(n)[0] + ".o"))
    with ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        list(ex.map(run, jobs))
    if _stale(BOUNDS_LIB, objs):
        run([nvcc, *ARCH, "-shared", "-o", BOUNDS_LIB, *objs])
    return BOUNDS_LIB


if __name__ == "__main__":
    print(build(verbose=True))

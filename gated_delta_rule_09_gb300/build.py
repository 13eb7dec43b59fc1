"""Build libgdn.so in place with nvcc for sm_103a (no cmake).

Each translation unit under ``csrc/`` compiles in parallel to an object in
``_build/``; the objects link into ``libgdn.so`` next to this file.  A source
or header newer than the library triggers a rebuild.

A second library, ``libgdn_waittest.so``, is the same code with the tensor-core
kernel compiled under ``GDN_WAIT_TEST``: 5 ms wait limits and one withheld
arrival in one unit, so the bounded-wait abort path can be run on purpose.
Only its test loads it; nothing else does.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgdn.so")
WAITTEST_LIB = os.path.join(PKG, "libgdn_waittest.so")
WAITTEST_SRC = "gdn_tc.cu"  # the translation unit the test build recompiles

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I" + INCLUDE, "-I" + CSRC, "--use_fast_math",
                     "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; libgdn needs the CUDA toolkit to build")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(INCLUDE, "gdn.h"),
                                                         os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(WAITTEST_LIB):
        return False
    t = min(os.path.getmtime(LIB), os.path.getmtime(WAITTEST_LIB))
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and not extra_flags and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    jobs = []
    for src in _sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        jobs.append((src, [cc, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]))
    wt_obj = os.path.join(BUILD, WAITTEST_SRC[:-3] + "_waittest.o")
    wt_src = os.path.join(CSRC, WAITTEST_SRC)
    jobs.append((wt_src, [cc, *NVCC_FLAGS, *extra_flags, "-DGDN_WAIT_TEST", "-c", wt_src, "-o", wt_obj]))
    for src, cmd in jobs:
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                            stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if out and (verbose or p.returncode):
            print(out, file=sys.stderr)
        if p.returncode:
            failed.append(os.path.basename(src))
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    wt_objs = [wt_obj if os.path.basename(o) == WAITTEST_SRC[:-3] + ".o" else o for o in objs]
    for lib, parts in ((WAITTEST_LIB, wt_objs), (LIB, objs)):
        tmp = lib + ".tmp.%d" % os.getpid()
        subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *parts], check=True)
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)

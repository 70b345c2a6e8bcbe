"""Build the CUDA library libfa_gb300.so in-tree (sm_103a only).

Each .cu under csrc/ is compiled in parallel with nvcc, then linked into one
shared library exposing the C ABI of include/fa.h.  No cmake, no torch
extension machinery: plain nvcc, so the same command works on any host that
has the CUDA 13 toolkit (x86_64 here, aarch64 on the GPU machines).

build(debug=True) makes the checked library libfa_gb300_debug.so instead
(-DFA_DEBUG=1: every TMA copy, TMEM access, hand-written shared-memory tile
store and work-item decode is checked against the rules of csrc/checks.h;
a broken rule is recorded in the device error word and the access skipped).
The package loads it when the environment sets FA_DEBUG=1.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(ROOT, "_build", "fa")
LIB = os.path.join(HERE, "libfa_gb300.so")
BUILD_DEBUG = os.path.join(ROOT, "_build", "fa_debug")
LIB_DEBUG = os.path.join(HERE, "libfa_gb300_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall", "-Xcompiler", "-fvisibility=hidden",
         "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hdrs + [os.path.join(ROOT, "include", "fa.h"), os.path.abspath(__file__)]


def _stale(target, inputs):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(x) > t for x in inputs)


def build(force: bool = False, verbose: bool = False, jobs: int | None = None, debug: bool = False) -> str:
    nvcc = _nvcc()
    bdir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    flags = FLAGS + (["-DFA_DEBUG=1"] if debug else [])
    os.makedirs(bdir, exist_ok=True)
    # objects and the library are host-architecture specific: rebuild everything
    # when the tree was last built on another kind of host
    stamp = os.path.join(bdir, "host.txt")
    host = platform.machine() + " " + nvcc
    if not os.path.exists(stamp) or open(stamp).read() != host or not os.path.exists(lib):
        force = True
    deps = _deps()
    srcs = _sources()
    objs = []
    todo = []
    for s in srcs:
        o = os.path.join(bdir, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or _stale(o, [s] + deps):
            todo.append((s, o))

    def compile_one(so):
        s, o = so
        cmd = [nvcc] + ARCH + flags + (["-Xptxas", "-v"] if verbose else []) + ["-c", s, "-o", o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s" % (s, r.stderr))
        return s, r.stderr

    if todo:
        with cf.ThreadPoolExecutor(max_workers=jobs or min(len(todo), os.cpu_count() or 4)) as ex:
            for s, err in ex.map(compile_one, todo):
                if verbose and err:
                    sys.stderr.write(err)
    if force or todo or _stale(lib, objs):
        tmp = lib + ".tmp.%d" % os.getpid()
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s" % r.stderr)
        os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(host)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))

"""Build the in-tree shared libraries with nvcc for sm_103a.

libfa.so           the attention library (C ABI in include/fa.h)
libfa_selftest.so  hardware self-checks (include/fa_selftest.h)
libfa_withhold.so  test build of libfa.so: every CTA leaves out one of its TMA copies
                   and waits give up after 20 ms, so that a test can check that the
                   kernels report FA_ERR_TIMEOUT and stop cleanly (not for any other use)
libfa_debug.so     libfa.so with bounds checks on every global, shared-memory and TMEM
                   access and TMA coordinate (include/fa_debug.h); slower, for tests

Each translation unit compiles in its own nvcc process, in parallel; objects
go to _build/ at the repository root. A library is rebuilt when any source or
header is newer than it.
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
BUILD = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I" + INCLUDE, "-I" + CSRC]

LIBS = {
    "libfa.so": ["fa_api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_noalloc.cu"],
    "libfa_selftest.so": ["selftest.cu"],
    "libfa_withhold.so": ["fa_api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_noalloc.cu"],
    "libfa_debug.so": ["fa_api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_noalloc.cu"],
}
# extra preprocessor definitions (and a separate object directory) per library
DEFINES = {
    "libfa_withhold.so": ["-DFA_TEST_WITHHOLD", "-DFA_WAIT_LIMIT_NS=20000000ull"],
    "libfa_debug.so": ["-DFA_DEBUG"],
}


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found")
    return p


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False) -> dict:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    headers = _headers()
    out = {}
    jobs = []
    plan = []
    for lib, srcs in LIBS.items():
        target = os.path.join(PKG, lib)
        srcs = [os.path.join(CSRC, s) for s in srcs]
        defs = DEFINES.get(lib, [])
        odir = os.path.join(BUILD, lib.replace(".so", "")) if defs else BUILD
        os.makedirs(odir, exist_ok=True)
        objs = [os.path.join(odir, os.path.basename(s) + ".o") for s in srcs]
        out[lib] = target
        if not force and not _stale(target, srcs + headers):
            continue
        for s, o in zip(srcs, objs):
            if force or _stale(o, [s] + headers):
                cmd = [cc] + ARCH + FLAGS + defs + ["-c", s, "-o", o]
                if verbose:
                    print(" ".join(cmd), flush=True)
                jobs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        plan.append((lib, target, objs))
    failed = []
    for cmd, p in jobs:
        so, _ = p.communicate()
        if p.returncode != 0:
            failed.append((cmd, so.decode(errors="replace")))
        elif verbose and so:
            print(so.decode(errors="replace"), flush=True)
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + log for c, log in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    for lib, target, objs in plan:
        tmp = target + ".tmp"
        cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
        os.replace(tmp, target)
    return out


if __name__ == "__main__":
    build(verbose="-v" in sys.argv, force="-f" in sys.argv)

"""Build ``libqd.so`` (the C-ABI decode library) in-tree with nvcc for sm_103a.

Translation units compile in parallel; the library links the CUDA runtime
statically so it loads without any Python package.  Outputs: ``libqd.so`` next
to this file and objects under ``_build/`` at the repository root.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libqd.so")
OBJDIR = os.path.join(ROOT, "_build", "qd")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def build(force: bool = False, verbose: bool = False, extra_flags=None, lib=None, objdir=None) -> str:
    """Compile every CUDA source for sm_103a and link ``libqd.so`` (or ``lib``, with its
    objects under ``objdir``: a variant build such as the phase-timeline one); returns
    the library's path."""
    LIB_ = lib or LIB
    OBJDIR_ = objdir or OBJDIR
    newest = max(os.path.getmtime(p) for p in _deps())
    if not force and os.path.exists(LIB_) and os.path.getmtime(LIB_) >= newest and not extra_flags:
        return LIB_
    os.makedirs(OBJDIR_, exist_ok=True)
    nvcc = _nvcc()
    flags = NVCC_FLAGS + list(extra_flags or [])
    procs = []
    objs = []
    for src in sources():
        obj = os.path.join(OBJDIR_, os.path.basename(src) + ".o")
        objs.append(obj)
        cmd = [nvcc] + ARCH + flags + ["-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((cmd, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"), file=sys.stderr)
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + o for c, o in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    tmp = LIB_ + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc] + ARCH + ["-shared", "-o", tmp] + objs)
    os.replace(tmp, LIB_)
    return LIB_


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

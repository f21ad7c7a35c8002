"""Build libgdnreplay.so in-tree with nvcc for sm_103a (GB300).

Run as ``python -m speculative_decode_recurrent_gb300.build``; the package's
``load()`` also calls :func:`build` when the library is missing or stale.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SOURCES = [os.path.join(PKG, "csrc", f)
           for f in ("gdn_replay.cu", "gdn_replay_tc.cu", "gdn_layer_ops.cu", "gdn_nonreplay.cu")]
HEADERS = [os.path.join(ROOT, "include", "gdnreplay.h"), os.path.join(ROOT, "include", "gdnlayer.h"),
           os.path.join(ROOT, "include", "gdnnonreplay.h"),
           os.path.join(PKG, "csrc", "replay_common.h"), os.path.join(PKG, "csrc", "tc_common.cuh")]
LIB = os.path.join(PKG, "_build", "libgdnreplay.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libgdnreplay cannot be built")


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in SOURCES + HEADERS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit in parallel, then link the shared library."""
    if not force and not stale():
        return LIB
    out = os.path.dirname(LIB)
    os.makedirs(out, exist_ok=True)
    common = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-I", os.path.join(ROOT, "include")]
    if verbose:
        common.append("-Xptxas=-v")
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(out, os.path.basename(src) + f".{os.getpid()}.o")
        objs.append(obj)
        procs.append(subprocess.Popen(common + ["-c", src, "-o", obj]))
    if any(p.wait() != 0 for p in procs):
        raise RuntimeError("nvcc failed while building libgdnreplay")
    tmp = LIB + f".{os.getpid()}.tmp"
    subprocess.check_call([nvcc(), *ARCH, "-shared", "-o", tmp, *objs])
    for o in objs:
        os.remove(o)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv))

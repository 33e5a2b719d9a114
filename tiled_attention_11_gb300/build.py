"""In-tree build of the CUDA libraries for sm_103a.

``libta11_fa.so`` is the attention library (include/fa.h); ``libta11_probe.so``
is the separate measurement library (csrc/probe.h: roof microbenchmarks and the
exp2 accuracy check), used only by the benchmark's tables and the tests.  Every
``csrc/*.cu`` translation unit is compiled by nvcc in parallel into ``_build/``;
the objects are linked into the package directory.  The CUDA runtime is linked
statically; the driver's tensor-map encoder is resolved at run time, so the
libraries load on a machine without a GPU (they then report FA_ERR_DEVICE on any
compute call).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libta11_fa.so")
SOURCES = ["fa_api.cu", "fwd_sm103a.cu", "bwd_sm103a.cu", "fwd_fp8_sm103a.cu", "quant_sm103a.cu"]
PROBE_LIB = os.path.join(PKG, "libta11_probe.so")
PROBE_SOURCES = ["probe_sm103a.cu"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest_input() -> float:
    t = 0.0
    for d in (CSRC, INCLUDE):
        for f in os.listdir(d):
            if f.endswith((".cu", ".cuh", ".h")):
                t = max(t, os.path.getmtime(os.path.join(d, f)))
    return max(t, os.path.getmtime(__file__))


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link both libraries if any source is newer than them; return the
    attention library's path."""
    os.makedirs(BUILD, exist_ok=True)
    newest = _newest_input()
    targets = [(LIB, SOURCES), (PROBE_LIB, PROBE_SOURCES)]
    stale = [(lib, srcs) for lib, srcs in targets
             if force or not os.path.exists(lib) or os.path.getmtime(lib) < newest]
    if not stale:
        return LIB
    nvcc = _nvcc()
    procs = []
    for _, srcs in stale:
        for src in srcs:
            obj = os.path.join(BUILD, src.replace(".cu", ".o"))
            cmd = [nvcc, *ARCH, *CFLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
                print(" ".join(cmd), file=sys.stderr)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    errors = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose and out:
            print(out, file=sys.stderr)
        if p.returncode != 0:
            errors.append(f"--- {src} ---\n{out}")
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    for lib, srcs in stale:
        objs = [os.path.join(BUILD, src.replace(".cu", ".o")) for src in srcs]
        tmp = lib + ".tmp"
        link = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
        r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout)
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

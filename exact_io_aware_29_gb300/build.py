"""Builds the CUDA library ``_build/libfa_gb300.so`` in-tree with nvcc for sm_103a.

Each translation unit compiles in its own nvcc process (in parallel), then one
shared library is linked with the CUDA runtime linked statically, so loading
it needs no libcuda on machines without a GPU. ``ptxas -v`` output (registers,
spills, shared memory per kernel) is kept next to the objects.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libfa_gb300.so")
SOURCES = ["api.cu", "fwd.cu", "bwd.cu", "decode.cu", "fp8.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "fa_gb300.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link; returns the library path. Raises on compiler errors."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                     "-I", os.path.join(ROOT, "include"), "-I", CSRC, "-Xptxas", "-v",
                     "--expt-relaxed-constexpr"]
    procs = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        log = open(os.path.join(BUILD, src.replace(".cu", ".ptxas.log")), "w")
        cmd = [cc, *common, "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log, obj))
    failed = []
    for src, p, log, _ in procs:
        p.wait()
        log.close()
        if p.returncode != 0:
            failed.append(src)
    if failed:
        msgs = []
        for src in failed:
            with open(os.path.join(BUILD, src.replace(".cu", ".ptxas.log"))) as f:
                msgs.append(f"--- {src}\n" + f.read()[-6000:])
        raise RuntimeError("nvcc failed:\n" + "\n".join(msgs))
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for *_, o in procs], "-cudart", "static"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    if verbose:
        for src in SOURCES:
            with open(os.path.join(BUILD, src.replace(".cu", ".ptxas.log"))) as f:
                sys.stdout.write(f.read())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

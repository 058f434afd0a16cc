"""Build the GB300 (sm_103a) shared library ``libgdn.so`` in-tree with nvcc.

Each translation unit compiles in parallel to ``_build/*.o`` with one
``-gencode`` (compute_103a / sm_103a); the objects link into
``hybrid_linear_attention_conv_gb300/libgdn.so`` with the CUDA runtime linked
statically, so the library needs nothing but the driver at load time.
``python -m hybrid_linear_attention_conv_gb300.build`` runs it by hand.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgdn.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")

SOURCES = ["gdn_api.cu", "gdn_decode.cu", "gdn_conv.cu", "gdn_prefill.cu", "gdn_snapshot.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "-I", INCLUDE, "-I", CSRC] + ARCH


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdn.so")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "gdn.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every CUDA source for sm_103a and link libgdn.so; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    procs = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        log = open(os.path.join(BUILD, src.replace(".cu", ".ptxas.log")), "w")
        cmd = [nvcc, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, obj, log, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT)))
    objs, failed = [], []
    for src, obj, log, proc in procs:
        proc.wait()
        log.close()
        if proc.returncode != 0:
            failed.append(src)
        objs.append(obj)
        if verbose or proc.returncode != 0:
            with open(log.name) as f:
                sys.stderr.write(f"--- {src}\n{f.read()}")
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([nvcc, "-shared", *ARCH, "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

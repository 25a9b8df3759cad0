"""Builds libtsp.so (the CUDA kernels + C ABI) in-tree for sm_103a.

Each .cu file compiles in parallel with nvcc; the objects are linked into
``folded_tensor_sequence_gb300/_build/libtsp.so``.  ptxas resource reports
(registers, spills, shared memory) land next to the objects as ``*.log``.
"""

from __future__ import annotations

import fcntl
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libtsp.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")

SOURCES = ["api.cu", "layout.cu", "gemm_simt.cu", "gemm_tc.cu", "attn_fwd.cu", "attn_fwd_tc.cu", "attn_bwd.cu", "attn_bwd_tc.cu", "attn_static.cu", "decode.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libtsp")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "tsp.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    # One build at a time (several processes may ask at once, e.g. parallel
    # test workers): the others wait on the lock and then find the library
    # up to date.
    with open(os.path.join(BUILD, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            if not force and up_to_date():
                return LIB
            return _compile(verbose)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def _compile(verbose: bool) -> str:
    nvcc = _nvcc()
    procs = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        log = open(os.path.join(BUILD, src.replace(".cu", ".log")), "w")
        cmd = [nvcc, *ARCH, *FLAGS, "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
    failed = []
    for src, p, log in procs:
        p.wait()
        log.close()
        if p.returncode != 0:
            failed.append(src)
    if failed:
        msgs = []
        for src in failed:
            with open(os.path.join(BUILD, src.replace(".cu", ".log"))) as f:
                msgs.append(f"--- {src}\n" + f.read()[-4000:])
        raise RuntimeError("nvcc failed:\n" + "\n".join(msgs))
    objs = [os.path.join(BUILD, s.replace(".cu", ".o")) for s in SOURCES]
    tmp = LIB + ".tmp"
    subprocess.run([nvcc, "-shared", *ARCH, "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}", file=sys.stderr)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)

"""Build the in-tree shared library ``libcb.so`` for sm_103a.

Each translation unit compiles in parallel with nvcc (host C++ with g++), then
nvcc links them with the static CUDA runtime.  The driver API is reached
through the runtime's entry-point query, so the library loads on a machine
without a GPU driver (only its host functions are usable there).
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libcb.so")
VALUES_SRC = os.path.join(PKG, "hostgen", "token_values.c")
VALUES_LIB = os.path.join(PKG, "libcb_values.so")

CUDA_SOURCES = ["runtime.cu", "append_kv.cu", "plan.cu", "split_kv.cu", "prefill_tc.cu", "attention.cu",
                "synth.cu", "decode_noalloc.cu", "selftest.cu", "decode_tc.cu"]
CXX_SOURCES = ["scheduler.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O3",
                     "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]
CXX_FLAGS = ["-O2", "-fPIC", "-std=c++17", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _cuda_include() -> str:
    return os.path.join(os.path.dirname(os.path.dirname(_nvcc())), "include")


def _fingerprint() -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            p = os.path.join(d, name)
            if os.path.isfile(p):
                h.update(name.encode())
                h.update(open(p, "rb").read())
    h.update(" ".join(NVCC_FLAGS + CXX_FLAGS).encode())
    h.update(__file__.encode())
    return h.hexdigest()


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build step failed ({r.returncode}):\n{' '.join(cmd)}\n{r.stdout}")
    return r.stdout


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if sources changed) and return the path of libcb.so."""
    stamp = os.path.join(BUILD, "fingerprint")
    fp = _fingerprint()
    if not force and os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == fp:
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    for src in CUDA_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        jobs.append(([nvcc, "-c", os.path.join(CSRC, src), "-o", obj] + NVCC_FLAGS, obj))
    for src in CXX_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        jobs.append((["g++", "-c", os.path.join(CSRC, src), "-o", obj, "-I", _cuda_include()]
                     + CXX_FLAGS, obj))
    workers = min(len(jobs), max(1, os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        list(ex.map(lambda j: _run(j[0], verbose), jobs))
    tmp = LIB + ".tmp"
    _run([nvcc, "-shared", "-o", tmp] + [o for _, o in jobs] + ARCH + ["-Xcompiler", "-fPIC"], verbose)
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(fp)
    return LIB


def build_values_lib(force: bool = False, verbose: bool = False) -> str:
    """Compile (if its source changed) the host-only input generator
    ``libcb_values.so`` with gcc and return its path.  It is separate from
    libcb.so and shares no source with it."""
    stamp = VALUES_LIB + ".fingerprint"
    h = hashlib.sha256(open(VALUES_SRC, "rb").read())
    h.update(__file__.encode())
    fp = h.hexdigest()
    if not force and os.path.exists(VALUES_LIB) and os.path.exists(stamp) and open(stamp).read() == fp:
        return VALUES_LIB
    tmp = VALUES_LIB + ".tmp"
    _run(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-o", tmp, VALUES_SRC, "-lm"],
         verbose)
    os.replace(tmp, VALUES_LIB)
    with open(stamp, "w") as f:
        f.write(fp)
    return VALUES_LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
    print(build_values_lib(force="--force" in sys.argv, verbose=True))

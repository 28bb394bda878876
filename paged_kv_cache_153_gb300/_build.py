"""Build libpkv.so and libpkv_prefill.so in-tree for sm_103a with nvcc (no
cmake, no torch extension).

The translation units compile in parallel.  Both shared libraries are linked
with the static CUDA runtime so they load without extra library paths.  The
prefill kernel (thread-block clusters sharing K/V loads by TMA multicast) sits
in libpkv_prefill.so of its own, so that a process that only decodes never
loads it; that library takes its error reporting from libpkv.so, found next to
it through an $ORIGIN run path.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libpkv.so")
PREFILL_LIB_PATH = os.path.join(PKG_DIR, "libpkv_prefill.so")

CUDA_SOURCES = ["append.cu", "api.cu", "decode_f16.cu", "decode_bf16.cu", "decode_e4m3.cu", "decode_e5m2.cu",
                "noalloc.cu", "decode_int8.cu", "append_int8.cu"]
PREFILL_SOURCES = ["prefill.cu"]
CXX_SOURCES = ["pool.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpkv.so")


def _source_digest() -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            if name.endswith((".cu", ".cuh", ".cpp", ".h")):
                with open(os.path.join(d, name), "rb") as f:
                    h.update(name.encode())
                    h.update(f.read())
    h.update(" ".join(ARCH + NVCC_FLAGS).encode())
    return h.hexdigest()


def _run(cmd: list[str]) -> None:
    res = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"build step failed ({res.returncode}): {' '.join(cmd)}\n{res.stdout}")


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libpkv.so and libpkv_prefill.so next to this file;
    skip when up to date."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    stamp = os.path.join(BUILD_DIR, "libpkv.stamp")
    digest = _source_digest()
    if not force and os.path.exists(LIB_PATH) and os.path.exists(PREFILL_LIB_PATH) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return LIB_PATH
    nvcc = _nvcc()
    jobs = []
    for src in CUDA_SOURCES + PREFILL_SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        jobs.append([nvcc, *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj])
    for src in CXX_SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cpp", ".o"))
        jobs.append([nvcc, *NVCC_FLAGS, "-x", "c++", "-c", os.path.join(CSRC, src), "-o", obj])
    with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        for cmd, _ in zip(jobs, ex.map(_run, jobs)):
            if verbose:
                print(" ".join(cmd))
    objs = [os.path.join(BUILD_DIR, s.rsplit(".", 1)[0] + ".o") for s in CUDA_SOURCES + CXX_SOURCES]
    tmp = LIB_PATH + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-Xlinker", "-soname,libpkv.so", "-o", tmp, *objs])
    os.replace(tmp, LIB_PATH)
    pobjs = [os.path.join(BUILD_DIR, s.rsplit(".", 1)[0] + ".o") for s in PREFILL_SOURCES]
    tmp = PREFILL_LIB_PATH + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *pobjs, "-L" + PKG_DIR, "-lpkv",
          "-Xlinker", "-rpath,$ORIGIN"])
    os.replace(tmp, PREFILL_LIB_PATH)
    with open(stamp, "w") as f:
        f.write(digest)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))

"""Builds the CUDA library libsgemm_gb300.so in-tree for sm_103a with nvcc.

Each translation unit is compiled in parallel, then linked into one shared
library under dense_fp32_sgemm_gb300/_build/.  A hash of the sources and
flags is stored next to it, so an unchanged tree is not rebuilt.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB_NAME = "libsgemm_gb300.so"
LIB_PATH = os.path.join(BUILD, LIB_NAME)

SOURCES = ["api.cu", "plan.cpp", "kernel_tile.cu", "kernel_skinny.cu", "kernel_generic.cu", "kernel_mid.cu",
           "kernel_ksplit.cu", "kernel_narrow.cu", "kernel_small.cu", "probes.cu", "noalloc.cu", "kernel_3xtf32.cu"]
HEADERS = ["device_common.cuh", "kernels.h", "kernels_3xtf32.h", "plan.h"]
PUBLIC_HEADERS = ["sgemm.h", "sgemm_probe.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
              "-Xptxas", "-v"]


def nvcc() -> str:
    cand = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cand, "bin", "nvcc")
    if os.path.exists(path):
        return path
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return found


def _digest() -> str:
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    for name in PUBLIC_HEADERS:
        with open(os.path.join(INCLUDE, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    h.update(" ".join(ARCH + NVCC_FLAGS).encode())
    return h.hexdigest()


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, "-x", "cu",
           "-c", os.path.join(CSRC, src), "-o", obj]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{proc.stdout}\n{proc.stderr}")
    return obj, proc.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if needed) and return the path of the shared library."""
    os.makedirs(BUILD, exist_ok=True)
    stamp = os.path.join(BUILD, "build.sha256")
    digest = _digest()
    if (not force and os.path.exists(LIB_PATH) and os.path.exists(stamp)
            and open(stamp).read().strip() == digest):
        return LIB_PATH
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as pool:
        results = list(pool.map(_compile, SOURCES))
    with open(os.path.join(BUILD, "ptxas.log"), "w") as log:
        for (obj, err), src in zip(results, SOURCES):
            log.write(f"== {src}\n{err}\n")
    tmp = LIB_PATH + ".tmp%d" % os.getpid()
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError(f"link failed:\n{proc.stdout}\n{proc.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(stamp, "w") as f:
        f.write(digest + "\n")
    if verbose:
        print(open(os.path.join(BUILD, "ptxas.log")).read())
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))

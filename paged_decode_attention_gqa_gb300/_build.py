"""Build libzl_decode_attn.so in-tree with nvcc for sm_103a.

Each .cu file is compiled in parallel into an object, then nvcc links them
into one shared library with the CUDA runtime linked statically (so the only
runtime dependency is the NVIDIA driver).
"""

from __future__ import annotations

import os
import shutil
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_DIR = os.path.join(HERE, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libzl_decode_attn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-diag-suppress", "1160", "-I", INCLUDE]

_lock = threading.Lock()


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    hdr = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hdr += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return sources() + hdr + [os.path.abspath(__file__)]


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(d) > t for d in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library if it is missing or older than its sources."""
    with _lock:
        if not force and not is_stale():
            return LIB_PATH
        os.makedirs(BUILD_DIR, exist_ok=True)
        os.makedirs(LIB_DIR, exist_ok=True)
        cc = nvcc()

        def compile_one(src):
            obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
            cmd = [cc, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
            if verbose and (r.stdout or r.stderr):
                print(r.stdout + r.stderr)
            return obj

        srcs = sources()
        with ThreadPoolExecutor(max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
            objs = list(ex.map(compile_one, srcs))
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB_PATH)
        return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))

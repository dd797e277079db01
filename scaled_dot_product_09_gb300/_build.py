"""Builds libsdpa09.so from csrc/ with nvcc for sm_103a, in-tree.

Each translation unit compiles in its own nvcc process (in parallel), then
one link step makes the shared library.  Outputs go to ``_build/`` next to
this file; a rebuild happens only when a source or header is newer than
the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libsdpa09.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
_lock = threading.Lock()


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsdpa09")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libsdpa09.so if it is missing or stale; return its path."""
    with _lock:
        if not force and not stale():
            return LIB
        os.makedirs(OUT, exist_ok=True)
        nvcc = nvcc_path()
        flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                        "-I" + INCLUDE, "--expt-relaxed-constexpr"]
        if verbose:
            flags += ["-Xptxas", "-v"]

        def compile_one(src):
            obj = os.path.join(OUT, os.path.basename(src)[:-3] + ".o")
            cmd = [nvcc] + flags + ["-c", src, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr[-4000:]}")
            return obj, r.stderr

        srcs = _sources()
        workers = max(1, min(len(srcs), os.cpu_count() or 4))
        with cf.ThreadPoolExecutor(workers) as ex:
            results = list(ex.map(compile_one, srcs))
        objs = [o for o, _ in results]
        if verbose:
            for _, log in results:
                print(log)
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
        os.replace(tmp, LIB)
        return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

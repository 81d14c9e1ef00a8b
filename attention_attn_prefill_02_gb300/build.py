"""Build the in-tree C-ABI shared library ``lib/libattn_gb300.so`` with nvcc for sm_103a.

Each translation unit under ``csrc/`` is compiled in parallel into ``_build/`` next to the
package, then linked with the static CUDA runtime (the library therefore loads on machines with
no GPU driver; every entry point then reports ATTN_ERR_NO_DEVICE).
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libattn_gb300.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
           "-Xcompiler", "-fvisibility=hidden"]
_lock = threading.Lock()


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _fingerprint() -> str:
    h = hashlib.sha256()
    for f in sorted(os.listdir(CSRC)) + ["attn.h"]:
        path = os.path.join(CSRC, f) if f != "attn.h" else os.path.join(INCLUDE, f)
        with open(path, "rb") as fh:
            h.update(f.encode() + fh.read())
    h.update(" ".join(ARCH + CUFLAGS).encode())
    return h.hexdigest()


def _compile(src: str, nvcc: str, verbose: bool) -> str:
    obj = os.path.join(OBJ, src + ".o")
    cmd = [nvcc, *ARCH, *CUFLAGS, "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose:
        print(r.stderr)
    return obj


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile (if sources changed) and return the path of the shared library."""
    with _lock:
        stamp = os.path.join(LIBDIR, ".fingerprint")
        fp = _fingerprint()
        if not force and os.path.exists(LIB) and os.path.exists(stamp):
            if open(stamp).read().strip() == fp:
                return LIB
        os.makedirs(OBJ, exist_ok=True)
        os.makedirs(LIBDIR, exist_ok=True)
        nvcc = _nvcc()
        srcs = _sources()
        with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
            objs = list(ex.map(lambda s: _compile(s, nvcc, verbose), srcs))
        tmp = LIB + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
        with open(stamp, "w") as fh:
            fh.write(fp)
        return LIB


if __name__ == "__main__":
    import sys

    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))

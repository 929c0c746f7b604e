"""Build libcsa.so in-tree with nvcc for sm_103a (GB300).

Each translation unit under csrc/ compiles to _build/<name>.o in parallel; the objects link
into compressed_sparse_attention_csa_gb300/libcsa.so against the shared CUDA runtime.
Rebuilds what is stale by modification time, and everything when the objects were built for
another host machine or another set of sources and flags (a stamp file records the machine
and a hash of the sources, headers and flags), so objects copied in from another machine are
never linked.  Usable as `python -m compressed_sparse_attention_csa_gb300.build`.
"""
from __future__ import annotations

import glob
import hashlib
import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(HERE, "libcsa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
                     "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcsa")
    return cand


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, verbose_ptxas: bool) -> str:
    obj = os.path.join(BUILD_DIR, os.path.splitext(os.path.basename(src))[0] + ".o")
    if _stale(obj, [src] + _headers()) or verbose_ptxas:
        cmd = [nvcc()] + NVCC_FLAGS + (["-Xptxas", "-v"] if verbose_ptxas else []) + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose_ptxas:
            sys.stderr.write(r.stderr)
    return obj


def _stamp(srcs) -> str:
    h = hashlib.sha256()
    h.update(platform.machine().encode())
    h.update(" ".join(NVCC_FLAGS).encode())
    for f in sorted(srcs) + sorted(_headers()):
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile every csrc/*.cu and link libcsa.so; returns the library path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    stamp_path = os.path.join(BUILD_DIR, "stamp.txt")
    stamp = _stamp(srcs)
    old = open(stamp_path).read().strip() if os.path.exists(stamp_path) else ""
    if force or old != stamp:
        for o in glob.glob(os.path.join(BUILD_DIR, "*.o")):
            os.remove(o)
        if os.path.exists(LIB_PATH):
            os.remove(LIB_PATH)
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas), srcs))
    if _stale(LIB_PATH, objs):
        cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", LIB_PATH] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    with open(stamp_path, "w") as fh:
        fh.write(stamp + "\n")
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))

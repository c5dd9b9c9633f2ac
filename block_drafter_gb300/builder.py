"""Builds ``_lib/libblockdrafter.so`` from ``csrc/*.cu`` for sm_103a (in-tree).

The translation units compile in parallel with nvcc and link into one shared library
exporting the C ABI declared in ``include/blockdrafter.h``.  A rebuild happens when any
source or header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "_lib")
LIBPATH = os.path.join(LIBDIR, "libblockdrafter.so")
OBJDIR = os.path.join(ROOT, "_build")
INCLUDE = os.path.join(ROOT, "include")

SOURCES = ["bd_abi.cu", "bd_gemm.cu", "bd_attention.cu", "bd_small.cu", "bd_noalloc.cu", "bd_pack.cu",
           "bd_head8.cu", "bd_bridge.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", "-Xptxas", "-v", f"-I{INCLUDE}"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)
             if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "blockdrafter.h"))
    return files


def is_stale() -> bool:
    if not os.path.exists(LIBPATH):
        return True
    t = os.path.getmtime(LIBPATH)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _compile(src: str) -> tuple:
    obj = os.path.join(OBJDIR, src.replace(".cu", ".o"))
    log = os.path.join(OBJDIR, src.replace(".cu", ".ptxas.txt"))
    cmd = [_nvcc()] + NVCC_FLAGS + ["-c", os.path.join(CSRC, src), "-o", obj]
    p = subprocess.run(cmd, capture_output=True, text=True)
    with open(log, "w") as f:
        f.write(p.stdout + p.stderr)
    return src, p.returncode, p.stdout + p.stderr, obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library if needed; returns its path.  Raises on failure."""
    if not force and not is_stale():
        return LIBPATH
    os.makedirs(OBJDIR, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    bad = [r for r in results if r[1] != 0]
    if bad:
        raise RuntimeError("nvcc failed:\n" + "\n".join(f"--- {r[0]}\n{r[2]}" for r in bad))
    if verbose:
        for r in results:
            sys.stdout.write(r[2])
    tmp = LIBPATH + ".tmp"
    cmd = [_nvcc()] + ARCH + ["-shared", "-Xcompiler", "-fPIC", "-o", tmp] + [r[3] for r in results]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError("link failed:\n" + p.stdout + p.stderr)
    os.replace(tmp, LIBPATH)
    return LIBPATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

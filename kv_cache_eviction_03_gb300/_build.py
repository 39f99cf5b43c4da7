"""Build the sm_103a C-ABI library `libh2o_gb300.so` in-tree with nvcc.

Each .cu translation unit compiles in parallel to an object file, then nvcc
links them into one shared library with the CUDA runtime linked statically.
Rebuilds only when a source or header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libh2o_gb300.so")
SOURCES = ["h2o_api.cu", "decode.cu", "prefill.cu", "select.cu", "noalloc.cu", "prefill_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA toolkit is required to build the H2O library")


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return files


def is_stale() -> bool:
    return is_stale_at(LIB)


def is_stale_at(path: str) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
          variant: str | None = None) -> str:
    """Compile the library if needed; returns its path.  `variant` builds a
    separately named copy (e.g. a profiling build with extra defines) next to
    the product library, with its own object files."""
    out_lib = LIB if variant is None else os.path.join(OUT_DIR, f"libh2o_gb300_{variant}.so")
    if not force and not is_stale_at(out_lib):
        return out_lib
    nvcc = _nvcc()
    obj_dir = OUT_DIR if variant is None else os.path.join(OUT_DIR, variant)
    os.makedirs(obj_dir, exist_ok=True)
    objs = []

    def compile_one(src: str) -> str:
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *(extra or []), "-I", INCLUDE, "-I", CSRC, "-c",
               os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = out_lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out_lib)
    return out_lib


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose=True))

"""Build the CUDA library in-tree: nvcc, one -gencode (sm_103a), translation
units compiled in parallel, then linked into ``_lib/libmoe_gb300.so``.

Run as ``python -m moe_routed_expert_gb300.build`` (or through
``__graft_entry__.build()``).  Rebuilds only when a source is newer than the
library.  ``--bounds`` (``build(bounds=True)``) builds the bounds-checking
variant ``_lib/libmoe_gb300_bounds.so`` (``-DMOE_BOUNDS_CHECK=1``: kernels
check the indexes they derive and report ``MOE_ERR_BOUNDS`` instead of
accessing out of range), which the binding loads when the environment sets
``MOE_GB300_BOUNDS_CHECK=1``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libmoe_gb300.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)
BOUNDS_LIB_PATH = os.path.join(OUT_DIR, "libmoe_gb300_bounds.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc_path() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hdrs + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]


def up_to_date(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(p) <= t for p in sources() + _deps() + [__file__])


def build(force: bool = False, verbose: bool = False, bounds: bool = False) -> str:
    lib_path = BOUNDS_LIB_PATH if bounds else LIB_PATH
    if not force and up_to_date(lib_path):
        return lib_path
    build_dir = BUILD_DIR + ("_bounds" if bounds else "")
    flags = NVCC_FLAGS + (["-DMOE_BOUNDS_CHECK=1"] if bounds else [])
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(build_dir, exist_ok=True)
    nvcc = nvcc_path()
    srcs = sources()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-lrt", "-ldl", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, bounds="--bounds" in sys.argv))

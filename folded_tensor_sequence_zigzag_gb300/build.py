"""Build libtsp.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Every .cu file under csrc/ is compiled in parallel to an object file under
_build/, then linked into folded_tensor_sequence_zigzag_gb300/libtsp.so.
Objects are rebuilt only when a source or header is newer.

    python -m folded_tensor_sequence_zigzag_gb300.build
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libtsp.so")
# checked build: every computed global index tested before its access
BUILD_CHECK = os.path.join(ROOT, "_build_check")
LIB_CHECK = os.path.join(PKG, "libtsp_check.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-I" + INCLUDE, "-I" + CSRC, "--expt-relaxed-constexpr"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (CUDA 13 toolkit required)")
    return cand


def _newest(paths):
    return max(os.path.getmtime(p) for p in paths)


def build(verbose: bool = False, jobs: int | None = None, check: bool = False) -> str:
    """libtsp.so, or with check=True libtsp_check.so (compiled with TSP_CHECK)."""
    out_dir, lib = (BUILD_CHECK, LIB_CHECK) if check else (BUILD, LIB)
    flags = NVCC_FLAGS + (["-DTSP_CHECK"] if check else [])
    os.makedirs(out_dir, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                     + glob.glob(os.path.join(INCLUDE, "*.h")))
    hdr_time = _newest(headers) if headers else 0.0
    objs, todo = [], []
    for src in sources:
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        objs.append(obj)
        if not os.path.exists(obj) or os.path.getmtime(obj) < max(os.path.getmtime(src), hdr_time):
            todo.append((src, obj))
    exe = nvcc()

    def compile_one(pair):
        src, obj = pair
        cmd = [exe, *ARCH, *flags, "-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stderr}")
        if verbose and res.stderr:
            print(res.stderr, file=sys.stderr)
        return obj

    if todo:
        with cf.ThreadPoolExecutor(max_workers=jobs or min(len(todo), os.cpu_count() or 4)) as ex:
            list(ex.map(compile_one, todo))
    if todo or not os.path.exists(lib) or os.path.getmtime(lib) < _newest(objs):
        tmp = lib + ".tmp"
        cmd = [exe, *ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64", "-o", tmp, *objs]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, check="--check" in sys.argv))

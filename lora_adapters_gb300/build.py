"""Build libslora.so in-tree for sm_103a (nvcc, no cmake).

Each translation unit is compiled in its own nvcc process, in parallel, then
linked with the static CUDA runtime into lora_adapters_gb300/libslora.so.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libslora.so")
# The SLORA_DEBUG build: the same sources with bounds checks in every kernel.
OBJ_DIR_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libslora_debug.so")
SOURCES = ["pool.cpp", "kernels.cu", "tc_kernels.cu", "noalloc.cu", "bmm.cu"]
HEADERS = [os.path.join(CSRC, "internal.h"), os.path.join(CSRC, "ptx.cuh"), os.path.join(ROOT, "include", "slora.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compiles libslora.so (debug: libslora_debug.so with -DSLORA_DEBUG)."""
    obj_dir, lib_path = (OBJ_DIR_DEBUG, LIB_DEBUG) if debug else (OBJ_DIR, LIB)
    if debug:
        extra_flags = (*extra_flags, "-DSLORA_DEBUG")
    os.makedirs(obj_dir, exist_ok=True)
    nvcc = _nvcc()
    srcs = [s for s in SOURCES if os.path.exists(os.path.join(CSRC, s))]
    jobs = []
    objs = []
    for s in srcs:
        src = os.path.join(CSRC, s)
        obj = os.path.join(obj_dir, s + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + HEADERS):
            xflags = ["-x", "cu"] if s.endswith(".cu") else []
            jobs.append([nvcc, *ARCH, *COMMON, *extra_flags, *xflags, "-c", src, "-o", obj])

    def run(cmd):
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        return subprocess.run(cmd, capture_output=True, text=True)

    with cf.ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        for cmd, res in zip(jobs, ex.map(run, jobs)):
            if res.returncode != 0:
                raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
            if verbose and res.stderr:
                print(res.stderr, file=sys.stderr)
    if force or jobs or _stale(lib_path, objs):
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static", "-ldl"]
        res = run(cmd)
        if res.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))

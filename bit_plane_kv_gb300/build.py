"""Build libfathom.so (the CUDA library behind include/fathom.h) in-tree.

One nvcc invocation per translation unit, run in parallel, for sm_103a only;
the objects are linked into ``bit_plane_kv_gb300/_build/libfathom.so``.
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
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libfathom.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfathom")


def _cuda_libdir(cc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(cc))), "lib64")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


DEBUG_LIB = os.path.join(OUT_DIR, "libfathom_debug.so")


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False, debug: bool = False) -> str:
    """Build libfathom.so, or with debug=True libfathom_debug.so: the same sources
    compiled with -DFATHOM_DEBUG, whose kernels check every data-derived index
    (see fathom_debug_status in include/fathom.h)."""
    out_dir = os.path.join(OUT_DIR, "debug") if debug else OUT_DIR
    lib_path = DEBUG_LIB if debug else LIB
    os.makedirs(out_dir, exist_ok=True)
    headers = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    srcs = sources()
    objs = [os.path.join(out_dir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    cc = nvcc()
    extra = ["-DFATHOM_DEBUG"] if debug else []

    def compile_one(src, obj):
        if not force and not _stale(obj, [src, *headers]):
            return ""
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        if ptxas_verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        return r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        logs = list(ex.map(lambda so: compile_one(*so), zip(srcs, objs)))
    if verbose or ptxas_verbose:
        for src, log in zip(srcs, logs):
            if log:
                sys.stderr.write(f"--- {os.path.basename(src)}\n{log}")
    if force or _stale(lib_path, objs):
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-rpath", "-Xlinker", _cuda_libdir(cc), "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv,
                debug="--debug" in sys.argv))

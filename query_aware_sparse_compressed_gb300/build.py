"""Build libqasc.so in-tree with nvcc for sm_103a.

Each .cu file in csrc/ compiles to an object under _build/ (in parallel,
skipped when newer than its source and every header), then nvcc links the
shared library next to this file.  The CUDA runtime is linked statically and
the driver API is reached through cudaGetDriverEntryPoint, so loading the
library needs no libcuda at link time.
"""

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libqasc.so")
# The instrumented variant: every entry point that enqueues work is an NVTX
# range named after it.  Separate objects and library, so the default build
# is never replaced by it.
NVTX_BUILD_DIR = os.path.join(PKG, "_build_nvtx")
NVTX_LIB = os.path.join(PKG, "libqasc_nvtx.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC,-fvisibility=hidden",
          "-I", INCLUDE, "-I", CSRC]


def nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand) and not shutil.which(cand):
        raise RuntimeError("nvcc not found; set NVCC or put the CUDA toolkit on PATH")
    return cand


def _headers():
    return (glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed (%d): %s\n%s%s" % (r.returncode, " ".join(cmd), r.stdout, r.stderr))
    return r


def build(force=False, verbose=False, jobs=None, nvtx=False):
    """Compile every kernel translation unit and link libqasc.so (with
    nvtx=True: libqasc_nvtx.so, built with -DQASC_NVTX).  Returns its path."""
    build_dir, lib = (NVTX_BUILD_DIR, NVTX_LIB) if nvtx else (BUILD_DIR, LIB)
    cflags = CFLAGS + (["-DQASC_NVTX"] if nvtx else [])
    os.makedirs(build_dir, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = _headers()
    cc = nvcc()
    jobs_todo = []
    objects = []
    for src in sources:
        obj = os.path.join(build_dir, os.path.splitext(os.path.basename(src))[0] + ".o")
        objects.append(obj)
        if force or _stale(obj, [src, *headers, __file__]):
            jobs_todo.append([cc, *cflags, "-c", src, "-o", obj])
    if jobs_todo:
        workers = jobs or min(len(jobs_todo), os.cpu_count() or 4)
        with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
            for f in [ex.submit(_run, cmd, verbose) for cmd in jobs_todo]:
                f.result()
    if force or jobs_todo or _stale(lib, objects):
        tmp = lib + ".tmp"
        _run([cc, "-shared", *ARCH, "-o", tmp, *objects, "-Xcompiler", "-fPIC"], verbose)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    path = build(force="--force" in sys.argv, verbose="-v" in sys.argv, nvtx="--nvtx" in sys.argv)
    print(path)

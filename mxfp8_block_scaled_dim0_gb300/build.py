"""Build ``libmxfp8_cast.so`` (the C ABI in include/mxfp8_cast.h) in-tree.

Each CUDA translation unit is compiled for sm_103a only, in parallel, then
linked into one shared library next to this file.  The CUDA runtime is linked
statically and the CUDA driver's tensor-map encoder is looked up at run time, so the
library loads on a machine without a GPU (for symbol checks).
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmxfp8_cast.so")
# Bounds-checked variant of the same sources (-DMX_DEBUG_BOUNDS): every global
# store the kernels issue is checked against its buffer (see mx_common.cuh);
# the tests run parity cases through it.
OBJ_DIR_BOUNDS = os.path.join(PKG, "_build_bounds")
LIB_BOUNDS = os.path.join(PKG, "libmxfp8_cast_bounds.so")
SOURCES = ["mx_cast.cu", "mx_blocked.cu", "mx_dequant.cu", "mx_scaled.cu", "mx_abi.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmxfp8_cast.so")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return files


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, verbose_ptxas=False, bounds=False):
    obj = os.path.join(OBJ_DIR_BOUNDS if bounds else OBJ_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-ftz=false", "-prec-div=true",
           "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, src),
           "-o", obj]
    if bounds:
        cmd.insert(1, "-DMX_DEBUG_BOUNDS")
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    return obj, r.stderr


def build(force: bool = False, verbose_ptxas: bool = False, bounds: bool = False) -> str:
    """Compile and link if any source is newer than the library.  bounds=True
    builds the bounds-checked variant (libmxfp8_cast_bounds.so) instead."""
    lib_path = LIB_BOUNDS if bounds else LIB
    deps = _deps()
    if not force and not verbose_ptxas and not _stale(lib_path, deps):
        return lib_path
    os.makedirs(OBJ_DIR_BOUNDS if bounds else OBJ_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose_ptxas, bounds), SOURCES))
    if verbose_ptxas:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib_path + ".tmp.%d" % os.getpid()
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                bounds="--bounds" in sys.argv))

"""Build libdllm.so (the CUDA path) in-tree for sm_103a.

Each ``csrc/*.cu`` (nvcc) and host-only ``csrc/*.cpp`` (g++) compiles to an
object in parallel; nvcc links them into
``block_decoding_gb300/libdllm.so`` against the CUDA runtime only (the one
driver call, the TMA tensor-map encoder, is fetched at run time through the
runtime's entry-point query, so the library loads on a machine without a
driver). Rebuilds only when a source or header is newer than the library.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdllm.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC] + ARCH


def _nvcc():
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else (shutil.which("nvcc") or "nvcc")


def _cuda_lib_dirs():
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    dirs = []
    for sub in ("lib64", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
        p = os.path.join(cuda, sub)
        if os.path.isdir(p):
            dirs.append(p)
            if os.path.isdir(os.path.join(p, "stubs")):
                dirs.append(os.path.join(p, "stubs"))
    return dirs


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return any(os.path.getmtime(p) > t for p in deps)


def _compile(src, extra):
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    if src.endswith(".cpp"):     # host-only runtime code
        cmd = [os.environ.get("CXX", "g++"), "-c", src, "-o", obj, "-O2", "-std=c++17", "-fPIC", "-Wall",
               "-I", INCLUDE, "-I", CSRC]
    else:
        cmd = [_nvcc(), "-c", src, "-o", obj] + NVCC_FLAGS + extra
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    """Compile every CUDA source and link libdllm.so; return its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    extra = list(extra_flags or [])
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda s: _compile(s, extra), sources()))
    if verbose:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    objs = [o for o, _ in results]
    tmp = LIB + ".tmp"
    link = [_nvcc(), "-shared", "-o", tmp] + objs + ARCH
    for dd in _cuda_lib_dirs():
        link += ["-L", dd]
    link += ["-lcudart"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    force = "--force" in sys.argv
    verbose = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None
    print(build(force=force or bool(extra), verbose=verbose or bool(extra), extra_flags=extra))

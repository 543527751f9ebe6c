"""Build the CUDA library in-tree: csrc/*.cu -> _build/libqmm_gb300.so (sm_103a only).

Each translation unit is compiled by its own nvcc process in parallel, then
linked into one shared library with the shared CUDA runtime.  build_variant()
builds the same sources with extra compile-time options (e.g. -DQMM_PAIR=1)
into another directory; a process started with QMM_GB300_LIB set to such a
library loads it instead of the in-tree one.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB_DEFAULT = os.path.join(BUILD, "libqmm_gb300.so")
LIB = os.environ.get("QMM_GB300_LIB") or LIB_DEFAULT
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build_library(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    if LIB != LIB_DEFAULT and os.path.exists(LIB):
        return LIB          # a variant chosen with QMM_GB300_LIB, built by its caller
    if not force and up_to_date():
        return LIB
    return _build(BUILD, LIB, NVCC_FLAGS + list(extra_flags or []), verbose)


def build_variant(extra_flags, out_dir: str, verbose: bool = False) -> str:
    """The library built with extra compile-time options into out_dir; returns its path."""
    os.makedirs(out_dir, exist_ok=True)
    return _build(out_dir, os.path.join(out_dir, "libqmm_gb300.so"), NVCC_FLAGS + list(extra_flags), verbose)


def _build(objdir: str, lib_path: str, flags, verbose: bool) -> str:
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *flags, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, _sources()))
    if verbose:
        for _, err in results:
            if err:
                print(err)
    objs = [o for o, _ in results]
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build_library(force=True, verbose="-v" in sys.argv))

"""Builds the in-tree CUDA library ``_build/libkda_gb300.so`` for sm_103a.

Each translation unit under ``csrc/`` is compiled by nvcc in parallel with
``-gencode arch=compute_103a,code=sm_103a -lineinfo -O3`` and linked with the
static CUDA runtime, so loading the library needs no libcudart on the path
(and loading it on a host without a GPU works; calling into the GPU does not).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libkda_gb300.so")
# tracing build: the same sources with the kernels' stage timers compiled in
# (-DKDA_STAGE_TIMERS), in a directory of its own
STAGE_BUILD = os.path.join(HERE, "_build_stage_timers")
STAGE_LIB = os.path.join(STAGE_BUILD, "libkda_gb300.so")
INCLUDE = os.path.join(ROOT, "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def build(force: bool = False, verbose: bool = False, extra_flags=(), stage_timers: bool = False) -> str:
    """Compiles the library (the tracing build with stage_timers=True) and
    returns its path."""
    out_dir, lib = (STAGE_BUILD, STAGE_LIB) if stage_timers else (BUILD, LIB)
    if stage_timers:
        extra_flags = (*extra_flags, "-DKDA_STAGE_TIMERS")
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    srcs = sources()
    newest_hdr = max(os.path.getmtime(h) for h in _headers())
    common = [nvcc, "-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC",
              "-I", INCLUDE, "-I", CSRC, *extra_flags]
    if verbose:
        common += ["-Xptxas", "-v"]

    def obj_of(src):
        return os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")

    def compile_one(src):
        obj = obj_of(src)
        if (not force and os.path.exists(obj)
                and os.path.getmtime(obj) >= max(os.path.getmtime(src), newest_hdr)):
            return obj, ""
        tmp = obj + f".tmp{os.getpid()}"
        r = subprocess.run(common + ["-c", src, "-o", tmp], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, obj)
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for _, log in results:
            if log:
                print(log)
    objs = [o for o, _ in results]
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs):
        tmp = lib + f".tmp{os.getpid()}"
        r = subprocess.run([nvcc, "-shared", *ARCH, "-cudart", "static", "-o", tmp, *objs],
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

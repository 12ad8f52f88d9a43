"""Builds libfdl.so in-tree with nvcc for sm_103a (GB300) only.

Each ``csrc/*.cu`` translation unit (and each host-only ``csrc/*.cpp`` one) is
compiled in parallel to an object under ``_build/`` and the objects are linked
into ``libfdl.so`` next to this file.
The CUDA runtime is linked statically, so the library depends only on the
driver at run time (the tensor-map encoder is fetched through the runtime's
driver entry-point query rather than by linking libcuda).
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfdl.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
         "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _obj(src: str) -> str:
    return os.path.join(OBJDIR, os.path.splitext(os.path.basename(src))[0] + ".o")


def build(verbose: bool = False, extra_flags=None) -> str:
    """Compiles (if needed) and returns the path of libfdl.so."""
    os.makedirs(OBJDIR, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    headers = sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")))
    flags = FLAGS + list(extra_flags or [])
    jobs = []
    for s in srcs:
        obj = _obj(s)
        if _stale(obj, [s, __file__] + headers):
            jobs.append((s, obj))

    def compile_one(job):
        s, obj = job
        cmd = [nvcc()] + ARCH + flags + ["-c", s, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(s)}:\n{r.stderr}")
        return s, r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for s, err in ex.map(compile_one, jobs):
            if verbose and err.strip():
                print(f"[{os.path.basename(s)}]\n{err}")
    objs = [_obj(s) for s in srcs]
    if jobs or _stale(LIB, objs):
        cmd = [nvcc()] + ARCH + ["-shared", "-o", LIB] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))

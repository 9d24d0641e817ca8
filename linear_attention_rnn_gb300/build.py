"""Builds libgdn.so (the C-ABI library) in-tree for sm_103a with nvcc.

Each .cu file under csrc/ is compiled in parallel to an object, then linked
into linear_attention_rnn_gb300/_build/libgdn.so.  Rebuilds only what is
older than its sources.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libgdn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                   "-I", CSRC] + list(extra)


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    newest_hdr = max((os.path.getmtime(h) for h in _headers()), default=0.0)
    jobs = []
    for s in srcs:
        obj = os.path.join(BUILD, os.path.basename(s)[:-3] + ".o")
        stale = (force or not os.path.exists(obj) or os.path.getmtime(obj) < os.path.getmtime(s)
                 or os.path.getmtime(obj) < newest_hdr)
        jobs.append((s, obj, stale))
    cmd0 = nvcc()
    extra = list(extra_flags) + (["-Xptxas", "-v"] if verbose else [])

    def compile_one(job):
        s, obj, stale = job
        if not stale:
            return ""
        r = subprocess.run([cmd0, *_flags(extra), "-c", s, "-o", obj], capture_output=True,
                           text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(s)}:\n{r.stderr}")
        return r.stderr

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        logs = list(ex.map(compile_one, jobs))
    if verbose:
        for lg in logs:
            if lg:
                print(lg)
    objs = [o for _, o, _ in jobs]
    if force or not os.path.exists(LIB) or any(os.path.getmtime(o) > os.path.getmtime(LIB) for o in objs):
        tmp = LIB + f".tmp{os.getpid()}"
        r = subprocess.run([cmd0, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs],
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

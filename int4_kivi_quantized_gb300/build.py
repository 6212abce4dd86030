"""Builds libs4kv.so in-tree with nvcc for sm_103a (no CMake, no torch extension)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libs4kv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]
# The quantizer must be IEEE-exact: no FMA contraction, IEEE division, no flush to zero.
EXACT = ["-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false"]
SOURCES = {
    "s4kv_host.cu": [],
    "s4kv_append.cu": EXACT,
    "s4kv_decode.cu": [],
    "s4kv_mq.cu": [],
    "s4kv_noalloc.cu": [],
}


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(obj: str, deps) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    # extra nvcc flags (e.g. -DS4KV_DECODE_WARPS=12) for tuning builds
    extra = tuple(extra) + tuple(os.environ.get("S4KV_EXTRA_NVCC", "").split())
    stamp = os.path.join(BUILD, "flags.txt")
    os.makedirs(BUILD, exist_ok=True)
    if not force and (not os.path.exists(stamp) or open(stamp).read() != " ".join(extra)):
        force = True
    with open(stamp, "w") as f:
        f.write(" ".join(extra))
    headers = [os.path.join(CSRC, "s4kv_common.cuh"), os.path.join(CSRC, "s4kv_kernels.cuh"),
               os.path.join(ROOT, "include", "s4kv.h"),
               __file__]
    jobs = []
    objs = []
    for src, flags in SOURCES.items():
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + headers):
            cmd = [nvcc(), *ARCH, *COMMON, *flags, *extra, "-c", s, "-o", o]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stderr

    logs = []
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            logs = list(ex.map(run, jobs))
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        r = subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"], capture_output=True,
                           text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    if verbose:
        for log in logs:
            print(log)
    return LIB


if __name__ == "__main__":
    import sys
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)

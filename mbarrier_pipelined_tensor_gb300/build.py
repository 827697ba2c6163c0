"""Builds libtp.so (the C-ABI library) in-tree with nvcc for sm_103a.

Every translation unit under csrc/ compiles in parallel to _build/*.o, then
one shared object is linked next to this file. A unit is rebuilt when it or
any header it may include is newer than its object. ``python -m
mbarrier_pipelined_tensor_gb300.build`` builds by hand.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libtp.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I", CSRC, "-I", INCLUDE]


def nvcc() -> str:
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    newest_header = max((os.path.getmtime(h) for h in _headers()), default=0.0)
    cc = nvcc()

    def obj_of(src):
        return os.path.join(BUILD, os.path.basename(src) + ".o")

    def needs(src):
        o = obj_of(src)
        return force or not os.path.exists(o) or os.path.getmtime(o) < max(os.path.getmtime(src), newest_header)

    def compile_one(src):
        cmd = [cc] + ARCH + FLAGS + ["-c", src, "-o", obj_of(src)]
        if src.endswith(".cpp"):
            cmd = [cc] + FLAGS + ["-x", "cu"] + ARCH + ["-c", src, "-o", obj_of(src)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        if verbose:
            print(os.path.basename(src), "ok", flush=True)

    # Objects of sources that no longer exist are removed: they are never
    # linked, and nothing stale should travel with the tree.
    live = {obj_of(s) for s in srcs}
    for o in glob.glob(os.path.join(BUILD, "*.o")):
        if o not in live:
            os.remove(o)
    todo = [s for s in srcs if needs(s)]
    if todo:
        with ThreadPoolExecutor(max(1, min(len(todo), os.cpu_count() or 1))) as ex:
            list(ex.map(compile_one, todo))
    objs = [obj_of(s) for s in srcs]
    if todo or not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        tmp = LIB + ".%d.tmp" % os.getpid()
        r = subprocess.run([cc] + ARCH + ["-shared", "-o", tmp] + objs, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stderr)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

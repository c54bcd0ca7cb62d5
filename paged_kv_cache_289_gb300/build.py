"""Build libpagedkv.so in-tree with nvcc for sm_103a (GB300).

Each .cu (device code) and .cpp (host-only code) under csrc/ is compiled to an
object in parallel by nvcc, then linked into
paged_kv_cache_289_gb300/lib/libpagedkv.so (CUDA runtime linked statically).
Objects are rebuilt when their source or any header is newer.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "libpagedkv.so")
INCLUDE = os.path.join(ROOT, "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc" if os.path.exists(
    "/usr/local/cuda/bin/nvcc") else "nvcc")


def _flags(verbose_ptxas: bool = False):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                "-Xcompiler", "-fvisibility=hidden"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    os.makedirs(LIBDIR, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    hdr_mtime = max([os.path.getmtime(h) for h in _headers()] + [0])
    objs = []
    todo = []
    for s in srcs:
        o = os.path.join(LIBDIR, os.path.splitext(os.path.basename(s))[0] + ".o")
        objs.append(o)
        if force or verbose_ptxas or not os.path.exists(o) or \
                os.path.getmtime(o) < max(os.path.getmtime(s), hdr_mtime):
            todo.append((s, o))

    def compile_one(so):
        s, o = so
        cmd = [NVCC] + _flags(verbose_ptxas) + ["-c", s, "-o", o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return s, r

    if todo:
        with ThreadPoolExecutor(max_workers=jobs or min(len(todo), os.cpu_count() or 4)) as ex:
            for s, r in ex.map(compile_one, todo):
                if verbose_ptxas or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed on {os.path.basename(s)}")
    if force or todo or not os.path.exists(LIB) or \
            os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [NVCC] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link of libpagedkv.so failed")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))

"""Build libringattn.so (sm_103a) in-tree with nvcc.

Each .cu translation unit compiles in parallel; the objects link into one
shared library next to this file.  Usage: ``python -m ring_attention_attn_gb300.build``.
``--checks`` builds the bounds-checked variant (``-DRA_CHECKS``: every kernel
checks the global row indices, TMA coordinates and TMEM columns it computes
and reports RA_ERR_BOUNDS instead of making an out-of-range access) into
``libringattn_checks.so``, with its objects in a build folder of its own;
load it through the RINGATTN_LIB environment variable.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libringattn.so")
BUILD_CHECKS = os.path.join(HERE, "_build_checks")
LIB_CHECKS = os.path.join(HERE, "libringattn_checks.so")
SOURCES = ["api.cu", "attn_bwd.cu", "attn_fwd.cu", "merge.cu", "noalloc.cu", "shard.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(verbose_ptxas: bool, checks: bool = False):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    if checks:
        f += ["-DRA_CHECKS"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None,
          checks: bool = False) -> str:
    build_dir, lib_path = (BUILD_CHECKS, LIB_CHECKS) if checks else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".cuh", ".h"))]
    headers.append(os.path.join(ROOT, "include", "ringattn.h"))
    objs, todo = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src[:-3] + ".o")
        objs.append(o)
        if force or verbose_ptxas or not _newer(o, [s] + headers):
            todo.append((s, o))
    cc = nvcc()

    def compile_one(so):
        s, o = so
        cmd = [cc] + _flags(verbose_ptxas, checks) + ["-c", s, "-o", o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return s, r

    if todo:
        with cf.ThreadPoolExecutor(max_workers=jobs or len(todo)) as ex:
            for s, r in ex.map(compile_one, todo):
                if verbose_ptxas or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed on {os.path.basename(s)}")
    if todo or not _newer(lib_path, objs):
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                checks="--checks" in sys.argv))

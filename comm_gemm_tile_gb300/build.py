"""Builds libmk.so in-tree with nvcc for sm_103a (GB300).

The library is plain CUDA C++ behind the C ABI in include/mk.h; each
translation unit compiles in parallel and the objects link with nvcc.
The same sources also build libmk_debug.so with MK_DEBUG_BOUNDS=1: device-side
index checks that report MK_ERR_INVALID instead of touching memory out of range.
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
LIB = os.path.join(HERE, "libmk.so")
LIB_DEBUG = os.path.join(HERE, "libmk_debug.so")
SOURCES = ["mk_api.cu", "mk_fused.cu", "mk_moe.cu", "mk_combine.cu", "mk_attn.cu", "mk_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def flags():
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                   "-I" + os.path.join(ROOT, "include"), "-I" + CSRC]


def _deps_mtime() -> float:
    t = 0.0
    for d in (CSRC, os.path.join(ROOT, "include")):
        for f in os.listdir(d):
            t = max(t, os.path.getmtime(os.path.join(d, f)))
    return t


def _fresh(lib: str) -> bool:
    return os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime()


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Build libmk.so (and with debug=True also libmk_debug.so, the
    bounds-checking build); returns the path of libmk.so.  Every translation
    unit of both libraries compiles in parallel."""
    targets = [(LIB, BUILD, [])]
    if debug:
        targets.append((LIB_DEBUG, os.path.join(BUILD, "debug"), ["-DMK_DEBUG_BOUNDS=1"]))
    todo = [t for t in targets if force or not _fresh(t[0])]
    if not todo:
        return LIB
    for _, d, _ in todo:
        os.makedirs(d, exist_ok=True)

    def compile_one(job):
        src, d, extra = job
        obj = os.path.join(d, src.replace(".cu", ".o"))
        cmd = [nvcc()] + flags() + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr, file=sys.stderr)
        return obj

    jobs = [(src, d, extra) for _, d, extra in todo for src in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(compile_one, jobs))
    for ti, (lib, _, _) in enumerate(todo):
        mine = objs[ti * len(SOURCES):(ti + 1) * len(SOURCES)]
        tmp = lib + ".tmp"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + mine + ["-lcudart_static", "-ldl", "-lpthread",
                                                                "-lrt"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))

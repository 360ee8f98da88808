"""Build libspecng.so in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in parallel into ``_build/`` at the repo
root, then linked into ``speculative_decoding_draft_ngram_gb300/libspecng.so``
(static CUDA runtime, no relocatable device code).  The same sources are
also built with ``-DSPECNG_CHECKED`` into ``libspecng_checked.so``: every
index computed from data is range-checked on the device (status bit
CHECKED_OOB, the index clamped, nothing trapped); load it with the
environment variable SPECNG_LIBRARY.  Run as
``python -m speculative_decoding_draft_ngram_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libspecng.so")
LIB_CHECKED = os.path.join(PKG, "libspecng_checked.so")
SOURCES = ["verify_bf16.cu", "verify_f32.cu", "lmhead.cu", "ngram.cu", "kv.cu", "capi.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecng")


def _stale(src_files, target) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(f) > t for f in src_files)


def build(verbose: bool = False, force: bool = False, extra_flags=(), checked: bool = True) -> str:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(ROOT, "include", "specng.h"))
    cc = nvcc()
    jobs = []
    variants = [(LIB, "", [])] + ([(LIB_CHECKED, "_checked", ["-DSPECNG_CHECKED"])] if checked else [])
    links = []
    for lib, tag, defs in variants:
        objs = []
        for src in SOURCES:
            s = os.path.join(CSRC, src)
            o = os.path.join(BUILD, src.replace(".cu", tag + ".o"))
            objs.append(o)
            if force or _stale([s] + headers, o):
                jobs.append([cc, *ARCH, *FLAGS, *defs, *extra_flags, "-c", s, "-o", o])
        links.append((lib, objs))

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        return r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        for out in ex.map(run, jobs):
            if verbose and out.strip():
                print(out, flush=True)
    for lib, objs in links:
        if force or jobs or _stale(objs, lib):
            run([cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", lib + ".tmp", *objs])
            os.replace(lib + ".tmp", lib)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))

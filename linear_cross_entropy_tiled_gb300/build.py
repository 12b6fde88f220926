"""Builds the CUDA library libflce.so in-tree for sm_103a (GB300).

    python -m linear_cross_entropy_tiled_gb300.build

Each .cu file under csrc/ compiles in parallel with nvcc. The objects are then
linked into linear_cross_entropy_tiled_gb300/lib/libflce.so, and compiled again with
FLCE_DEBUG (every kernel store checked against its buffer) into
lib/libflce_debug.so. Each .cu file under
probes/ (stand-alone measurement programs, not part of the library) becomes an
executable lib/flce_probe_<name>. nvcc cross-compiles, so this also works on a
machine without a GPU.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
PROBES = os.path.join(PKG, "probes")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libflce.so")
DEBUG_LIB = os.path.join(LIBDIR, "libflce_debug.so")   # FLCE_DEBUG: checked stores
BUILD = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libflce.so")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def probe_sources() -> list[str]:
    return sorted(os.path.join(PROBES, f) for f in os.listdir(PROBES) if f.endswith(".cu"))


def probe_path(src: str) -> str:
    return os.path.join(LIBDIR, "flce_probe_" + os.path.basename(src)[:-3])


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + probe_sources()
    files.append(os.path.join(INCLUDE, "flce.h"))
    return max(os.path.getmtime(f) for f in files)


def up_to_date() -> bool:
    outs = [LIB, DEBUG_LIB] + [probe_path(p) for p in probe_sources()]
    return all(os.path.exists(o) and os.path.getmtime(o) >= _deps_mtime() for o in outs)


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    cc = nvcc()
    extra = extra or []

    def compile_one(job: tuple[str, bool]) -> str:
        src, debug = job
        obj = os.path.join(BUILD, os.path.basename(src) + (".debug.o" if debug else ".o"))
        cmd = [cc, *ARCH, *FLAGS, *extra, *(["-DFLCE_DEBUG"] if debug else []), "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    def build_probe(src: str) -> str:
        exe = probe_path(src)
        r = subprocess.run([cc, *ARCH, "-O3", "-lineinfo", "-std=c++17", *extra, src, "-o", exe],
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        return exe

    srcs = sources()
    probes = probe_sources()
    jobs = [(src, False) for src in srcs] + [(src, True) for src in srcs]
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(jobs) + len(probes)) as ex:
        probe_jobs = [ex.submit(build_probe, p) for p in probes]
        objs = list(ex.map(compile_one, jobs))
        for j in probe_jobs:
            j.result()
    for out, part in ((LIB, objs[:len(srcs)]), (DEBUG_LIB, objs[len(srcs):])):
        tmp = out + ".tmp"
        r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *part], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, out)
    return LIB


if __name__ == "__main__":
    force = "--force" in sys.argv
    verbose = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None
    print(build(force=force, verbose=verbose or bool(extra), extra=extra))

"""Build libpgqa.so in-tree with nvcc for sm_103a (GB300).

Each .cu file under csrc/ is compiled to an object in parallel, then the
objects are linked into ``libpgqa.so`` beside this file. The CUDA runtime is
linked statically, so the library needs only the driver at run time.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpgqa.so")
# the same library with the split kernel's per-phase %globaltimer stamps
# compiled in (see timeline.py); never built by default
BUILD_TIMELINE = os.path.join(HERE, "_build_timeline")
LIB_TIMELINE = os.path.join(HERE, "libpgqa_timeline.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpgqa")
    return exe


def _flags(verbose_ptxas: bool, timeline: bool = False) -> list[str]:
    f = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC, *ARCH]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    if timeline:
        f += ["-DPGQA_TIMELINE"]
    return f


def _sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "pgqa.h"))
    return files


def _compile(src: str, verbose_ptxas: bool, timeline: bool = False) -> tuple[str, str]:
    obj = os.path.join(BUILD_TIMELINE if timeline else BUILD, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *_flags(verbose_ptxas, timeline), "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose_ptxas: bool = False, timeline: bool = False) -> str:
    """Compile and link libpgqa.so (timeline=True: libpgqa_timeline.so, the
    same sources with the per-phase stamps); returns its path. Skips work
    when up to date."""
    lib = LIB_TIMELINE if timeline else LIB
    if not force and not verbose_ptxas and os.path.exists(lib):
        newest = max(os.path.getmtime(p) for p in _deps())
        if os.path.getmtime(lib) >= newest:
            return lib
    os.makedirs(BUILD_TIMELINE if timeline else BUILD, exist_ok=True)
    srcs = _sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose_ptxas, timeline), srcs))
    if verbose_ptxas:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))

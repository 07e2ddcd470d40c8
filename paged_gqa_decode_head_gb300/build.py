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
# Measurement builds of the same sources, never built by default:
# "timeline" compiles in the split kernel's per-phase %globaltimer stamps
# (see timeline.py).
VARIANTS = {
    "timeline": ("-DPGQA_TIMELINE", "libpgqa_timeline.so"),
}


def _variant_paths(variant):
    if variant is None:
        return BUILD, LIB
    define, name = VARIANTS[variant]
    return os.path.join(HERE, "_build_" + variant), os.path.join(HERE, name)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpgqa")
    return exe


def _flags(verbose_ptxas: bool, variant=None) -> list[str]:
    f = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC, *ARCH]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    if variant is not None:
        f += [VARIANTS[variant][0]]
    return f


def _sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "pgqa.h"))
    return files


def _compile(src: str, verbose_ptxas: bool, variant=None) -> tuple[str, str]:
    obj = os.path.join(_variant_paths(variant)[0], os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *_flags(verbose_ptxas, variant), "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose_ptxas: bool = False, variant: str | None = None) -> str:
    """Compile and link libpgqa.so (or a measurement build named in
    VARIANTS); returns its path. Skips work when up to date."""
    build_dir, lib = _variant_paths(variant)
    if not force and not verbose_ptxas and os.path.exists(lib):
        newest = max(os.path.getmtime(p) for p in _deps())
        if os.path.getmtime(lib) >= newest:
            return lib
    os.makedirs(build_dir, exist_ok=True)
    srcs = _sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose_ptxas, variant), srcs))
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

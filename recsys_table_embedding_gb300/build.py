"""Build the CUDA library libtbe_gb300.so in-tree for sm_103a (GB300).

Each translation unit under csrc/ is compiled by nvcc in parallel, then the
objects are linked into one shared library next to this file.  Objects go to
_build/ (git-ignored).  Set TBE_PTXAS_VERBOSE=1 to print ptxas register and
shared-memory reports.
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
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libtbe_gb300.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtbe_gb300.so")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")] + [
        os.path.join(INCLUDE, "tbe.h")]


STAMP = os.path.join(BUILD, "flags.txt")


def _flags() -> list:
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                    "-I", CSRC, "--expt-relaxed-constexpr", "-Xcompiler", "-Wall"]
    # tuning knobs (-DTBE_FWD_ROWS=...), e.g. for launch-shape sweeps
    return flags + os.environ.get("TBE_NVCC_DEFINES", "").split()


def up_to_date() -> bool:
    """The library exists, is newer than every source, and was built with the
    same compiler flags (tuning knobs included)."""
    if not os.path.exists(LIB) or not os.path.exists(STAMP):
        return False
    if open(STAMP).read() != " ".join(_flags()):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    flags = _flags()
    if os.environ.get("TBE_PTXAS_VERBOSE"):
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, "-c", src, "-o", obj] + flags
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or os.environ.get("TBE_PTXAS_VERBOSE"):
            sys.stderr.write(r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = [nvcc, "-shared", "-o", tmp] + objs + ARCH + ["-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(" ".join(_flags()))
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

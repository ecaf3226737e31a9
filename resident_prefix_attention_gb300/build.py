"""Builds the replay-attention library ``liblsr.so`` in-tree for sm_103a.

Each CUDA translation unit is compiled in parallel with nvcc, then linked
into one shared library next to this file.  Objects go to ``_build/``.

With the environment variable ``LSR_DEBUG=1`` the kernels are built with
their bounds checks (an output index outside its buffer sets
``LSR_DEV_BOUNDS`` in the pool's status word and the access is skipped);
the build records its flags and rebuilds when they change.
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
LIB = os.path.join(HERE, "liblsr.so")
SOURCES = ["lsr_api.cu", "kernels_mem.cu", "attn_fwd.cu", "attn_bwd.cu",
           "profile.cu", "noalloc.cu", "selftest.cu",
           "score.cu", "window.cu", "group.cu", "latent.cu",
           "latent_bwd.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC",
         "-I" + os.path.join(ROOT, "include")] + ARCH
STAMP = os.path.join(BUILD, "flags")


def _flags():
    debug = os.environ.get("LSR_DEBUG", "") not in ("", "0")
    return FLAGS + (["-DLSR_DEBUG"] if debug else [])


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build")


def _deps():
    inc = os.path.join(ROOT, "include")
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(inc, f) for f in os.listdir(inc)
              if f.endswith(".h")]
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(STAMP):
        return False
    with open(STAMP) as f:
        if f.read() != " ".join(_flags()):
            return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if needed) and return the path of liblsr.so."""
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    flags = _flags()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", obj] + flags
        if verbose:
            cmd.append("-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp"
    cmd = [nvcc, "-shared", "-o", tmp] + objs + ARCH
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(" ".join(flags))
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

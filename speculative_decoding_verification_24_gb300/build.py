"""In-tree build of libspecverify.so (sm_103a only).

Each CUDA source compiles to an object in parallel, then nvcc links the
shared library next to this file. The CUDA runtime is linked statically, so
the library loads on a machine without a GPU (for the ABI tests) and needs
nothing but the driver on a machine with a GPU.

The same sources also build libspecverify_debug.so with SPECVERIFY_DEBUG
defined: the verify kernel then checks every global load and store against
the buffers of the call and reports an access outside them (which it skips)
in the status word, without trapping.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libspecverify.so")
LIB_DEBUG = os.path.join(PKG, "libspecverify_debug.so")
# (library, object directory, extra flags)
VARIANTS = [(LIB, BUILD_DIR, []), (LIB_DEBUG, os.path.join(BUILD_DIR, "debug"), ["-DSPECVERIFY_DEBUG"])]

SOURCES = ["verify_logits.cu", "verify_grouped.cu", "lmhead.cu", "prompt_lookup.cu", "api.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "specverify.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    for lib, _, _ in VARIANTS:
        if not os.path.exists(lib):
            return False
        t = os.path.getmtime(lib)
        if not all(os.path.getmtime(f) <= t for f in _inputs()):
            return False
    return True


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libspecverify.so and libspecverify_debug.so; returns
    the path of the first."""
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()

    def compile_one(job):
        src, obj_dir, extra = job
        obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    jobs = []
    for _, obj_dir, extra in VARIANTS:
        os.makedirs(obj_dir, exist_ok=True)
        jobs += [(src, obj_dir, extra) for src in SOURCES]
    with ThreadPoolExecutor(len(jobs)) as pool:
        objs = list(pool.map(compile_one, jobs))
    for k, (lib, _, _) in enumerate(VARIANTS):
        tmp = lib + f".tmp{os.getpid()}"
        mine = objs[k * len(SOURCES):(k + 1) * len(SOURCES)]
        r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *mine], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

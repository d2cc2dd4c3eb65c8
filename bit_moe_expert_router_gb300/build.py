"""In-tree build of the package's native libraries.

``libmoe_w4a8.so``: the CUDA kernels and the C ABI, compiled by nvcc for
sm_103a only (one -gencode), one translation unit per source file, in
parallel.  ``synth/libsynth.so``: the seeded input generator (plain C).
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
REPO = os.path.dirname(PKG)
INCLUDE = os.path.join(REPO, "include")
LIB = os.path.join(PKG, "libmoe_w4a8.so")
SYNTH_LIB = os.path.join(PKG, "synth", "libsynth.so")
OBJ_DIR = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]
C_FLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed: " + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def _newer(target: str, sources) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(s) <= t for s in sources)


def build_synth(force: bool = False) -> str:
    src = os.path.join(PKG, "synth", "synth.c")
    if force or not _newer(SYNTH_LIB, [src]):
        _run(["gcc", *C_FLAGS, "-o", SYNTH_LIB, src, "-lm"])
    return SYNTH_LIB


def cuda_sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def build_cuda(force: bool = False, verbose_ptxas: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(OBJ_DIR, exist_ok=True)
    srcs = cuda_sources()
    headers = _headers()
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []

    def compile_one(src):
        obj = os.path.join(OBJ_DIR, os.path.basename(src) + ".o")
        if force or verbose_ptxas or not _newer(obj, [src, *headers]):
            return obj, _run([nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj])
        return obj, ""

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(compile_one, srcs))
    objs = [o for o, _ in results]
    if force or not _newer(LIB, objs):
        _run([nvcc, *ARCH, "-shared", "-o", LIB, *objs])
    if verbose_ptxas:
        return "\n".join(log for _, log in results)
    return LIB


def build(force: bool = False) -> None:
    build_synth(force)
    build_cuda(force)

"""Build the C-ABI library ``_build/libpod_attn.so`` in-tree with nvcc for sm_103a only.

Two translation units (the CUDA kernels + C ABI, and the host planner) compile in parallel,
then nvcc links them with the static CUDA runtime. The driver API entry point the library needs
(tensor-map encoding) is looked up at run time, so the library loads on hosts without a GPU.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libpod_attn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = [os.path.join(CSRC, f) for f in ("pod_attn.cu", "planner.cpp")]
HEADERS = [os.path.join(CSRC, f) for f in ("pod_internal.h", "ptx.cuh")] + [
    os.path.join(os.path.dirname(HERE), "include", "pod_attn.h")]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in SOURCES + HEADERS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if sources changed) and return the path of libpod_attn.so."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC"] + ARCH

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src) + f".{os.getpid()}.o")
        cmd = [nvcc] + common + ["-c", src, "-o", obj]
        if src.endswith(".cu"):
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if src.endswith(".cu"):
            with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
                f.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs, capture_output=True,
                       text=True)
    for o in objs:
        os.remove(o)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        print(open(os.path.join(BUILD, "ptxas.log")).read())
    return LIB

"""Build the C-ABI library libpadecode.so in-tree with nvcc for sm_103a.

Each CUDA source compiles in parallel to an object under _build/, then the
objects link into paged_kv_attention_15_gb300/libpadecode.so. Sources that
did not change since their object was made are not recompiled.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libpadecode.so")

SOURCES = ["pa_api.cu", "pa_inst_bf16.cu", "pa_inst_f16.cu", "pa_inst_fp8.cu", "pa_inst_umma.cu",
           "pa_inst_umma_fp8.cu", "pa_inst_qrow.cu", "pa_inst_pair.cu", "pa_append.cu"]
HEADERS = ["pa_ptx.cuh", "pa_kernels.cuh", "pa_reduce.cuh", "pa_launch.h", "pa_inst_bf16.cu", "pa_tc.cuh",
           "pa_umma.cuh", "pa_inst_umma.cu", "pa_qrow.cuh", "pa_pair.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpadecode.so")


def _flags(verbose_ptxas: bool) -> list:
    f = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC] + ARCH
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [src] + [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "pa_decode.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose_ptxas: bool = False, force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    jobs = []
    objs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(BUILD, s.replace(".cu", ".o"))
        objs.append(obj)
        if force or verbose_ptxas or _stale(obj, src):
            jobs.append([cc, "-c", src, "-o", obj] + _flags(verbose_ptxas))
    logs = []
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for cmd, res in zip(jobs, ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs)):
            logs.append(res.stdout + res.stderr)
            if res.returncode != 0:
                raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    if jobs or force or not os.path.exists(LIB) or any(os.path.getmtime(o) > os.path.getmtime(LIB) for o in objs):
        cmd = [cc, "-shared", "-o", LIB] + objs + ARCH + ["-lcudart"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("link failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    if verbose_ptxas:
        sys.stdout.write("\n".join(logs))
    return LIB


if __name__ == "__main__":
    build(verbose_ptxas="-v" in sys.argv, force="--force" in sys.argv)
    print(LIB)

"""Build the in-tree shared library ``_build/libpk.so`` with nvcc for sm_103a.

Four translation units: the host planner (``csrc/pk_plan.cpp``), the
attention kernel plus launcher (``csrc/pk_attn.cu``), the LSE merge
(``csrc/pk_merge.cu``) and the host-buffer pipeline (``csrc/pk_pipeline.cpp``).  They compile in parallel and are linked against the
shared CUDA runtime (the one PyTorch loads too).
"""
from __future__ import annotations

import hashlib
import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libpk.so")
SOURCES = ["pk_plan.cpp", "pk_attn.cu", "pk_merge.cu", "pk_pipeline.cpp"]
HEADERS = [os.path.join(CSRC, "pk_internal.h"), os.path.join(CSRC, "tmem_ops.cuh"),
           os.path.join(CSRC, "sync.cuh"), os.path.join(CSRC, "attn_common.cuh"),
           os.path.join(INCLUDE, "pk.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found")
    return found


STAMP = LIB + ".stamp"


def _fingerprint() -> str:
    """Host architecture + the bytes of every source and header: a library
    built elsewhere (another machine type) or from other sources is stale,
    whatever the file times say."""
    h = hashlib.sha256(platform.machine().encode())
    for p in [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [__file__]:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _stale() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(STAMP):
        return True
    with open(STAMP) as f:
        return f.read().strip() != _fingerprint()


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, src + f".{os.getpid()}.o")
        cmd = [cc, *ARCH, "-lineinfo", *common, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose_ptxas and src.endswith(".cu"):
            cmd.insert(1, "-Xptxas=-v")
        subprocess.run(cmd, check=True)
        return obj

    objs = [os.path.join(BUILD, src + f".{os.getpid()}.o") for src in SOURCES]
    tmp = LIB + f".tmp{os.getpid()}"
    try:
        with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
            list(ex.map(compile_one, SOURCES))
        subprocess.run([cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs], check=True)
        os.replace(tmp, LIB)
    finally:
        for o in objs + [tmp]:
            if os.path.exists(o):
                os.remove(o)
    with open(STAMP, "w") as f:
        f.write(_fingerprint())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))

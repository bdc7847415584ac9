"""Build libsvdq.so in-tree: the sm_103a CUDA kernels (nvcc) plus the host
packers (g++, no fused multiply-add so the packed codes are deterministic),
linked with the static CUDA runtime so that loading the library needs no GPU
driver.  ``python -m bit_w4a4_diffusion_quantize_b300.build`` rebuilds what is
out of date."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libsvdq.so")
INCLUDE = os.path.join(ROOT, "include")

CUDA_SOURCES = ["capi.cu", "quantize_act.cu", "gemm_w4a4.cu", "gemm_int4.cu", "awq_gemv.cu",
                "microbench.cu", "selftest.cu"]
HOST_SOURCES = ["pack.cpp"]
HEADERS = ["device_common.cuh", "act_quant.cuh", "int4_quant.cuh", "launch.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsvdq")


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    if verbose and (r.stdout.strip() or r.stderr.strip()):
        print(r.stdout + r.stderr, flush=True)
    return r


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile every source that changed and link libsvdq.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "svdq.h"),
                                                       os.path.join(INCLUDE, "svdq_bench.h"),
                                                       os.path.join(INCLUDE, "svdq_test.h")]
    objs = []
    for src in CUDA_SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src + ".o")
        objs.append(o)
        if force or ptxas_info or _newer(o, [s, __file__] + hdrs):
            cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-I", INCLUDE, "-c", s, "-o", o]
            if ptxas_info:
                cmd += ["-Xptxas", "-v"]
            r = _run(cmd, verbose)
            if ptxas_info:
                print(r.stderr, flush=True)
    for src in HOST_SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src + ".o")
        objs.append(o)
        if force or _newer(o, [s, __file__] + hdrs):
            _run(["g++", "-O3", "-std=c++17", "-fPIC", "-ffp-contract=off", "-pthread",
                  "-march=x86-64-v2", "-I", INCLUDE, "-c", s, "-o", o], verbose)
    if force or _newer(LIB, objs):
        tmp = LIB + ".tmp"
        _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs,
              "-Xcompiler", "-pthread"], verbose)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)

"""Builds ``libconv2d_gb300.so`` in-tree with nvcc for sm_103a.

Translation units compile in parallel; the result is linked with the static CUDA
runtime so that the library needs nothing but the driver at load time.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libconv2d_gb300.so")

SOURCES = ["conv_tap_gemm.cu", "conv_wgrad.cu", "conv_wgrad_mn.cu", "conv_dgrad_c2i.cu", "conv_depthwise.cu", "conv3d_copy.cu", "conv2d_api.cpp",
           "conv3d_api.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA toolkit is required to build the library")


def _stale(srcs, target) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in srcs)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile (if needed) and return the path of the shared library."""
    os.makedirs(OUT_DIR, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "conv2d_gb300.h"))
    nvcc = _nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I", INCLUDE, "-I", CSRC] + list(extra_flags)
    jobs = []
    objs = []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(OUT_DIR, src + ".o")
        objs.append(obj)
        if force or _stale([path] + headers, obj):
            cmd = [nvcc] + common + ["-c", path, "-o", obj]
            if src.endswith(".cu"):
                cmd += ["-Xptxas", "-v"] if verbose else []
            jobs.append(cmd)

    def run(cmd):
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("compile failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
        return res.stdout + res.stderr

    logs = []
    if jobs:
        with concurrent.futures.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            logs = list(ex.map(run, jobs))
    if force or jobs or _stale(objs, LIB):
        tmp = LIB + f".tmp{os.getpid()}"
        run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static"])
        os.replace(tmp, LIB)
    if verbose:
        for lg in logs:
            print(lg)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

"""Planner invariants on the host (no GPU): compiles tests/planner_check.cpp against the
library's planner source and its built kernel objects (for the shared-memory size functions)
and runs it; it plans the three ops for workloads, test shapes, dilated and grouped problems
and checks the budgets, ring sizes, tap coverage, that every tap of every forward and
backward-data pass reads the source pixel the definition names, the pass counts of large
filters, and the exactly-once production of every (channel, tap) of the filter gradient."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "convolution_nchw_conv2d_gb300", "csrc")
OBJS = os.path.join(ROOT, "convolution_nchw_conv2d_gb300", "_build")


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def test_planner_invariants(tmp_path):
    import __graft_entry__
    __graft_entry__.build()  # leaves the kernel objects in _build/
    cuda = _cuda_home()
    objs = [os.path.join(OBJS, n) for n in ("conv_tap_gemm.cu.o", "conv_wgrad.cu.o", "conv_wgrad_mn.cu.o", "conv_dgrad_c2i.cu.o", "conv_depthwise.cu.o")]
    if not all(os.path.exists(o) for o in objs):
        pytest.skip("kernel objects not found next to the built library")
    exe = str(tmp_path / "planner_check")
    cmd = ["g++", "-O1", "-std=c++17", "-I", os.path.join(cuda, "include"), "-I", os.path.join(ROOT, "include"),
           "-I", CSRC, os.path.join(ROOT, "tests", "planner_check.cpp")] + objs + \
          ["-L", os.path.join(cuda, "lib64"), "-L", os.path.join(cuda, "lib64", "stubs"), "-lcudart", "-lcuda",
           "-lpthread", "-ldl", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    env = dict(os.environ)
    env["LD_LIBRARY_PATH"] = os.path.join(cuda, "lib64") + ":" + env.get("LD_LIBRARY_PATH", "")
    r = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert "0 violations" in r.stdout

"""The allocation-free forward entry point, conv2d_fwd_noalloc.

Some callers cannot allocate device memory: their memory belongs to another runtime's
pool, or they run on a path that must never call cudaMalloc (it can synchronize the
device).  conv2d_fwd_noalloc serves them by staging the repacked filter in a fixed 8 MiB
scratch array inside the library instead of a caller workspace.  These tests call it
through the C ABI and check the results against the fp64 oracle within the TF32 / bf16
tolerances of the parity tests: two different problems in a row (the second must not see
the first one's staged filter), a filter large enough to run as several tap passes, a
problem whose staged filter is exactly the 8 MiB limit (accepted), and two beyond it
(refused).  This file is collected last and passes both alone and after the other tests.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from convolution_nchw_conv2d_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
LIMIT = 8 << 20


def _noalloc_via_cabi(lib, pb, x, w):
    y = torch.full(pb.y_shape, float("nan"), dtype=x.dtype, device=DEV)
    dt = 0 if pb.dtype == "f32" else 1
    stream = torch.cuda.current_stream()
    rc = lib.conv2d_fwd_noalloc(*pb.dims(), dt, ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    return rc, y


def _fwd_workspace(lib, pb):
    size = ctypes.c_size_t(0)
    assert lib.conv2d_workspace_size(0, *pb.dims(), 0 if pb.dtype == "f32" else 1, ctypes.byref(size)) == 0
    return size.value


def _check_oracle(pb, got, x, w, what):
    got = got.double().cpu().numpy()
    assert np.all(np.isfinite(got)), f"{what}: unwritten output element"
    ref = oracle.conv2d_fwd(x, w, (pb.pad_h, pb.pad_w), (pb.stride_h, pb.stride_w))
    if pb.dtype == "f32":
        tol = 2e-3 * math.sqrt(pb.C * pb.R * pb.S) * float(x.abs().max()) * float(w.abs().max())
        err = float(np.abs(got - ref).max())
        assert err <= tol, f"{what}: max|err| {err:.3e} > {tol:.3e}"
    else:
        rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
        assert rel <= 1e-2, f"{what}: relative-to-norm error {rel:.3e}"


def _run_and_check(lib, cg, pb, x, w, what):
    rc, y = _noalloc_via_cabi(lib, pb, x.to(DEV), w.to(DEV))
    assert rc == 0, f"{what}: conv2d_fwd_noalloc returned {rc} ({cg.conv2d_strerror(rc)})"
    cg.conv2d_device_status()
    _check_oracle(pb, y, x, w, what)


def test_noalloc_forward_matches_oracle_twice():
    import convolution_nchw_conv2d_gb300 as cg
    lib = cg.load_library()
    # Two consecutive calls share the library's scratch: the second must not see the
    # first call's packed filter.
    for name in ("resnet3x3", "deconv"):
        wl = W.WORKLOADS[name]
        x, w, _ = W.make_inputs(wl)
        _run_and_check(lib, cg, wl.problem, x, w, name)


def test_noalloc_large_filter_in_tap_passes():
    """A 16x16 filter over 32 channels: conv2d_fwd runs it as two tap passes adding onto y."""
    import convolution_nchw_conv2d_gb300 as cg
    lib = cg.load_library()
    pb = W.Conv2dProblem(1, 32, 40, 40, 32, 16, 16, 7, 7, 1, 1)
    x, w, _ = W.random_problem_inputs(pb, 9900)
    _run_and_check(lib, cg, pb, x, w, "16x16 filter")


def test_noalloc_accepts_exactly_the_limit():
    import convolution_nchw_conv2d_gb300 as cg
    lib = cg.load_library()
    # 1x1, C = 2048, K = 1024, fp32: the repacked filter is 1024 x 2048 x 4 bytes = 8 MiB, and
    # conv2d_fwd stages this fp32 x directly (no channel-chunk copy), so its workspace is the filter.
    pb = W.Conv2dProblem(1, 2048, 4, 4, 1024, 1, 1)
    assert _fwd_workspace(lib, pb) == LIMIT
    x, w, _ = W.random_problem_inputs(pb, 9901)
    _run_and_check(lib, cg, pb, x, w, "8 MiB filter")


@pytest.mark.parametrize("C,K", [(2048, 1025), (2048, 2048)])
def test_noalloc_rejects_filters_beyond_its_scratch(C, K):
    import convolution_nchw_conv2d_gb300 as cg
    lib = cg.load_library()
    # 1x1: one more output channel than the limit holds (a whole extra tile), and 16 MiB.
    pb = W.Conv2dProblem(1, C, 4, 4, K, 1, 1)
    assert _fwd_workspace(lib, pb) > LIMIT
    x = torch.zeros(pb.x_shape, device=DEV)
    w = torch.zeros(pb.w_shape, device=DEV)
    y = torch.zeros(pb.y_shape, device=DEV)
    rc = lib.conv2d_fwd_noalloc(*pb.dims(), 0, ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                ctypes.c_void_p(y.data_ptr()), None)
    assert rc == -13
    assert "scratch" in cg.conv2d_strerror(rc)

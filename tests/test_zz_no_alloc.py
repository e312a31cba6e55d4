"""The allocation-free forward entry point, conv2d_fwd_noalloc.

Some callers cannot allocate device memory (their memory belongs to another runtime's
pool, or they run on a path that must never call cudaMalloc).  conv2d_fwd_noalloc serves
them by staging the repacked filter in a fixed scratch array inside the library instead
of a caller workspace.  This test calls it through the C ABI twice in a row, on different
problems, and checks each result against the regular conv2d_fwd (which takes a
workspace) within the TF32 / bf16 tolerances the parity tests use.  It lives in its own
file, collected last, and passes both alone and after the other tests.
"""
import ctypes
import math

import pytest
import torch

from convolution_nchw_conv2d_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _noalloc_via_cabi(lib, pb, x, w):
    y = torch.full(pb.y_shape, float("nan"), dtype=x.dtype, device=DEV)
    dt = 0 if pb.dtype == "f32" else 1
    stream = torch.cuda.current_stream()
    rc = lib.conv2d_fwd_noalloc(*pb.dims(), dt, ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0, f"conv2d_fwd_noalloc returned {rc}"
    return y


def _close(pb, got, ref, x, w):
    assert not torch.isnan(got).any().item()
    g, r = got.double(), ref.double()
    if pb.dtype == "f32":
        tol = 2e-3 * math.sqrt(pb.C * pb.R * pb.S) * float(x.abs().max()) * float(w.abs().max())
        assert float((g - r).abs().max()) <= tol
    else:
        assert float((g - r).norm()) <= 1e-2 * float(r.norm())


def test_noalloc_forward_matches_workspace_forward_twice():
    import convolution_nchw_conv2d_gb300 as cg
    lib = cg.load_library()
    # Two consecutive calls share the library's scratch: the second must not see the
    # first call's packed filter.
    for name in ("resnet3x3", "deconv"):
        wl = W.WORKLOADS[name]
        pb = wl.problem
        x, w, _ = W.make_inputs(wl)
        xd, wd = x.to(DEV), w.to(DEV)
        got = _noalloc_via_cabi(lib, pb, xd, wd)
        ref = cg.conv2d_fwd(xd, wd, (pb.pad_h, pb.pad_w), (pb.stride_h, pb.stride_w))
        cg.conv2d_device_status()
        _close(pb, got, ref, x, w)


def test_noalloc_rejects_filters_beyond_its_scratch():
    import convolution_nchw_conv2d_gb300 as cg
    lib = cg.load_library()
    # 1x1, C = K = 2048: the repacked fp32 filter needs 16 MiB > 8 MiB.
    pb = W.Conv2dProblem(1, 2048, 4, 4, 2048, 1, 1)
    x = torch.zeros(pb.x_shape, device=DEV)
    w = torch.zeros(pb.w_shape, device=DEV)
    y = torch.zeros(pb.y_shape, device=DEV)
    rc = lib.conv2d_fwd_noalloc(*pb.dims(), 0, ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                ctypes.c_void_p(y.data_ptr()), None)
    assert rc == -13
    assert "scratch" in cg.conv2d_strerror(rc)

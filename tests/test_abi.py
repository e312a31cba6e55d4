"""C-ABI checks that need no GPU: the library loads, exports every symbol the header
declares, validates descriptors on the host, sizes workspaces, and links no vendor
convolution/GEMM library."""
import ctypes
import os
import re
import subprocess

import pytest

import oracle
from convolution_nchw_conv2d_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "conv2d_gb300.h")


@pytest.fixture(scope="module")
def cg():
    import __graft_entry__
    __graft_entry__.build()
    import convolution_nchw_conv2d_gb300 as m
    return m


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|int|unsigned\s+long\s+long)\s*(conv[23]d_\w+)\s*\(", text,
                                 re.M)))


def test_header_declares_the_abi():
    names = _declared()
    for n in ("conv2d_fwd", "conv2d_bwd_data", "conv2d_bwd_filter", "conv2d_workspace_size",
              "conv2d_output_dim", "conv2d_strerror", "conv2d_device_status", "conv2d_fwd_noalloc",
              "conv2d_kernel_launches", "conv3d_workspace_size", "conv3d_fwd", "conv3d_bwd_data",
              "conv3d_bwd_filter", "conv2d_bwd"):
        assert n in names


def test_library_exports_every_declared_symbol(cg):
    lib = ctypes.CDLL(cg.lib_path())
    for n in _declared():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", cg.lib_path()], capture_output=True, text=True).stdout
    for n in _declared():
        assert re.search(rf"\bT {n}\b", out), n


def test_no_vendor_conv_or_gemm_library_linked(cg):
    out = subprocess.run(["nm", "-D", cg.lib_path()], capture_output=True, text=True).stdout.lower()
    deps = subprocess.run(["ldd", cg.lib_path()], capture_output=True, text=True).stdout.lower()
    for bad in ("cudnn", "cublas", "dnnl", "mkldnn"):
        assert bad not in out and bad not in deps


def test_output_dim_matches_oracle(cg):
    for inp in range(1, 40):
        for pad in range(0, 4):
            for k in range(1, 8):
                for st in range(1, 4):
                    want = oracle.output_dim(inp, pad, k, st)
                    if want >= 1:
                        assert cg.conv2d_output_dim(inp, pad, k, st) == want
                    else:
                        with pytest.raises(cg.Conv2dError):
                            cg.conv2d_output_dim(inp, pad, k, st)


def _ws(cg, op, dims, dt=0):
    lib = cg.load_library()
    out = ctypes.c_size_t(0)
    rc = lib.conv2d_workspace_size(op, *dims, dt, ctypes.byref(out))
    return rc, out.value


GOOD = (2, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1, 8, 8)


@pytest.mark.parametrize("bad,code", [
    ((0, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1, 8, 8), -1),    # N = 0
    ((2, 3, 8, 8, 4, 3, 3, -1, 1, 1, 1, 8, 8), -1),   # negative pad
    ((2, 3, 8, 8, 4, 3, 3, 1, 1, 0, 1, 8, 8), -1),    # stride 0
    ((2, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1, 7, 8), -2),    # P mismatch
    ((2, 3, 2, 8, 4, 5, 3, 0, 1, 1, 1, 0, 8), -2),    # no output rows
    ((65536, 256, 256, 256, 4, 3, 3, 1, 1, 1, 1, 256, 256), -7),  # too large
    ((1, 1, 80, 80, 1, 65, 65, 0, 0, 1, 1, 16, 16), -11),  # R*S > 4096 (16 passes of 256 taps)
    ((1, 1, 90, 90, 1, 9, 9, 0, 0, 9, 9, 10, 10), -11),    # stride_h*stride_w > 64
])
def test_descriptor_errors(cg, bad, code):
    for op in (0, 1, 2):
        rc, _ = _ws(cg, op, bad)
        assert rc == code
    lib = cg.load_library()
    dummy = ctypes.c_void_p(0x1000)
    for fn in (lib.conv2d_fwd, lib.conv2d_bwd_data, lib.conv2d_bwd_filter):
        assert fn(*bad, 0, dummy, dummy, dummy, None, 0, None) == code


def test_bad_dtype_and_op(cg):
    assert _ws(cg, 0, GOOD, dt=7)[0] == -5
    assert _ws(cg, 9, GOOD)[0] == -12
    lib = cg.load_library()
    assert lib.conv2d_workspace_size(0, *GOOD, 0, None) == -3


def test_null_and_misaligned_pointers(cg):
    lib = cg.load_library()
    p = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10002)
    for fn in (lib.conv2d_fwd, lib.conv2d_bwd_data, lib.conv2d_bwd_filter):
        assert fn(*GOOD, 0, None, p, p, None, 0, None) == -3
        assert fn(*GOOD, 0, odd, p, p, None, 0, None) == -4


def test_workspace_sizes_are_bounded(cg):
    for wl in W.WORKLOADS.values():
        pb = wl.problem
        dt = 0 if pb.dtype == "f32" else 1
        for op in (0, 1, 2):
            rc, n = _ws(cg, op, pb.dims(), dt)
            assert rc == 0 and 0 <= n <= 1_000_000_000 and n % 16 == 0
            # fp32 backward-data with few input channels runs without a workspace
            few = op == 1 and pb.dtype == "f32" and pb.C <= 8
            assert (n == 0) == few, (wl.name, op, n)


def test_strided_filter_gradient_workspace_stays_under_the_cap(cg):
    """Strided backward-filter may stage a copy of x in the workspace (stride phases); a layer
    whose x alone passes the 1e9-byte cap runs without it, so the size stays under the cap."""
    x_over_cap = (112, 256, 96, 96, 256, 3, 3, 1, 1, 2, 2, 48, 48)  # x: 1.06e9 bytes in fp32
    rc, n = _ws(cg, 2, x_over_cap, 0)
    assert rc == 0 and 0 < n <= 1_000_000_000
    strided = W.WORKLOADS["strided"].problem  # takes the phases: x (102.8 MB) is in the size
    rc, n = _ws(cg, 2, strided.dims(), 0)
    assert rc == 0 and n > strided.N * strided.C * strided.H * strided.W * 4


def test_strerror_covers_codes(cg):
    for c in range(0, -13, -1):
        assert cg.conv2d_strerror(c) and "unknown error" not in cg.conv2d_strerror(c)


# ------------------------------------------------------------------ extended entry points
def _ws_ex(cg, op, dims, dil=(1, 1), groups=1, dt=0):
    lib = cg.load_library()
    out = ctypes.c_size_t(0)
    rc = lib.conv2d_workspace_size_ex(op, *dims, dil[0], dil[1], groups, dt, ctypes.byref(out))
    return rc, out.value


def test_ex_entry_points_validate_on_the_host(cg):
    """Mode, dilation and groups are checked before anything is planned or launched."""
    lib = cg.load_library()
    d = ctypes.c_void_p(0x10000)
    grp = (2, 6, 8, 8, 9, 3, 3, 1, 1, 1, 1, 8, 8)
    # unknown mode
    assert lib.conv2d_fwd_ex(*GOOD, 1, 1, 1, 0, 2, d, d, None, ctypes.c_float(0), d, None, 0, None) == -1
    assert lib.conv2d_bwd_data_ex(*GOOD, 1, 1, 1, 0, 5, d, d, None, ctypes.c_float(0), d, None, 0, None) == -1
    assert lib.conv2d_bwd_filter_ex(*GOOD, 1, 1, 1, 0, -1, d, d, ctypes.c_float(0), d, None, None, None, 0,
                                    None) == -1
    # dilation < 1
    assert _ws_ex(cg, 0, GOOD, dil=(0, 1))[0] == -1
    # P, Q must follow the dilated filter extent: R = 3, dilation 2 -> extent 5
    assert _ws_ex(cg, 0, GOOD, dil=(2, 2))[0] == -2
    assert _ws_ex(cg, 0, (2, 3, 8, 8, 4, 3, 3, 2, 2, 1, 1, 8, 8), dil=(2, 2))[0] == 0
    # groups must divide C and K
    assert _ws_ex(cg, 0, grp, groups=3)[0] == 0
    assert _ws_ex(cg, 0, grp, groups=2)[0] == -1      # K = 9
    assert _ws_ex(cg, 2, grp, groups=0)[0] == -1
    for op in (0, 1, 2):
        assert _ws_ex(cg, op, GOOD)[1] == _ws(cg, op, GOOD)[1]   # defaults = the plain sizing


def test_grouped_and_dilated_workspace_bounded(cg):
    for dims, dil, groups in [((32, 64, 56, 56, 64, 3, 3, 1, 1, 1, 1, 56, 56), (1, 1), 2),
                              ((32, 64, 56, 56, 64, 3, 3, 2, 2, 1, 1, 56, 56), (2, 2), 1),
                              ((8, 32, 28, 28, 32, 3, 3, 1, 1, 1, 1, 28, 28), (1, 1), 32)]:
        for op in (0, 1, 2):
            rc, n = _ws_ex(cg, op, dims, dil, groups)
            assert rc == 0 and 0 <= n <= 1_000_000_000 and n % 16 == 0
            # backward-data with few input channels per group, and the forward and backward-data
            # of depthwise layers (one input channel per group), run without a workspace
            depthwise = groups > 1 and dims[1] // groups == 1
            assert (n == 0) == ((op == 1 and dims[1] // groups <= 8) or (op == 0 and depthwise)), (dims, op, n)

"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Tolerances (fixed by the workload definition):
  fp32 tensors (TF32 tensor cores): max|err| <= 2e-3 * sqrt(L) * max|a| * max|b|, with
      a, b the op's two inputs and L the number of products in the longest sum the op
      forms: C*R*S (forward), K*ceil(R/stride_h)*ceil(S/stride_w) (backward-data: an input
      pixel is reached by at most ceil(R/stride_h) filter rows and ceil(S/stride_w) filter
      columns) and N*P*Q (backward-filter).  The literal C*R*S form is also enforced for
      the forward op.
  bf16 tensors: ||err||_2 / ||ref||_2 <= 1e-2, the oracle run on the bf16 inputs.
Every output is pre-filled with NaN, so an element the kernels fail to write fails
the test; a second run must reproduce the first bit for bit.  The six workloads are
compared element by element against the full oracle; when the environment variable
CONV2D_PARITY_REPORT names a file, one line per (workload, op) with max|err| / tol (or the
relative-to-norm error for bf16) is appended to it.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from convolution_nchw_conv2d_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def cg():
    import convolution_nchw_conv2d_gb300 as m
    m.load_library()
    return m


def _poisoned(shape, dtype):
    return torch.full(shape, float("nan"), dtype=dtype, device=DEV)


def _run(cg, op, pb, x, w, dy):
    pad, st = (pb.pad_h, pb.pad_w), (pb.stride_h, pb.stride_w)
    if op == "fwd":
        out = _poisoned(pb.y_shape, x.dtype)
        cg.conv2d_fwd(x, w, pad, st, out=out)
    elif op == "bwd_data":
        out = _poisoned(pb.x_shape, x.dtype)
        cg.conv2d_bwd_data(dy, w, (pb.H, pb.W), pad, st, out=out)
    else:
        out = _poisoned(pb.w_shape, x.dtype)
        cg.conv2d_bwd_filter(x, dy, (pb.R, pb.S), pad, st, out=out)
    cg.conv2d_device_status()
    return out


def _red_len(op, pb):
    """Products in the longest sum of the op (dilation 1)."""
    rows = -(-pb.R // pb.stride_h)
    cols = -(-pb.S // pb.stride_w)
    return {"fwd": pb.C * pb.R * pb.S, "bwd_data": pb.K * rows * cols, "bwd_filter": pb.N * pb.P * pb.Q}[op]


def _operands(op, x, w, dy):
    return {"fwd": (x, w), "bwd_data": (dy, w), "bwd_filter": (x, dy)}[op]


def _oracle_full(op, pb, x, w, dy):
    pad, st = (pb.pad_h, pb.pad_w), (pb.stride_h, pb.stride_w)
    if op == "fwd":
        return oracle.conv2d_fwd(x, w, pad, st)
    if op == "bwd_data":
        return oracle.conv2d_bwd_data(dy, w, (pb.H, pb.W), pad, st)
    return oracle.conv2d_bwd_filter(x, dy, (pb.R, pb.S), pad, st)


def _check(op, pb, got, ref, a, b, what):
    """Asserts the tolerance; returns the ratio of the error to its bound (<= 1 passes)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} != {ref.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite output (unwritten element?)"
    err = np.abs(got - ref)
    amax = float(a.abs().max()) if a.numel() else 0.0
    bmax = float(b.abs().max()) if b.numel() else 0.0
    if pb.dtype == "f32":
        tol = 2e-3 * math.sqrt(_red_len(op, pb)) * amax * bmax
        e = float(err.max(initial=0.0))
        assert e <= tol, f"{what}: max|err| {e:.3e} > {tol:.3e}"
        if op == "fwd":
            lit = 2e-3 * math.sqrt(pb.C * pb.R * pb.S) * amax * bmax
            assert e <= lit
        return e / tol if tol > 0 else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref)) / den if den > 0 else float(np.linalg.norm(got))
    assert rel <= 1e-2, f"{what}: relative-to-norm error {rel:.3e} > 1e-2"
    return rel / 1e-2


def _report(line):
    path = os.environ.get("CONV2D_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(line + "\n")


# ------------------------------------------------------------------ the six workloads
OPS = ["fwd", "bwd_data", "bwd_filter"]


_ORACLE_CACHE = {}


def _oracle_cached(op, name, pb, x, w, dy):
    key = (name, op)
    if key not in _ORACLE_CACHE:
        _ORACLE_CACHE.clear()  # one full-size result at a time (the large ones are hundreds of MB)
        _ORACLE_CACHE[key] = _oracle_full(op, pb, x, w, dy)
    return _ORACLE_CACHE[key]


@pytest.mark.parametrize("name", list(W.WORKLOADS))
@pytest.mark.parametrize("op", OPS)
def test_workload_parity(cg, name, op):
    """Every output element of every workload against the full fp64 oracle."""
    wl = W.WORKLOADS[name]
    pb = wl.problem
    x, w, dy = W.make_inputs(wl)
    xd, wd, dyd = x.to(DEV), w.to(DEV), dy.to(DEV)
    out = _run(cg, op, pb, xd, wd, dyd)
    assert not torch.isnan(out).any().item(), "unwritten output elements"
    a, b = _operands(op, x, w, dy)
    ref = _oracle_cached(op, name, pb, x, w, dy)
    ratio = _check(op, pb, out.double().cpu().numpy(), ref, a, b, f"{name}/{op}")
    kind = "max|err|/tol" if pb.dtype == "f32" else "rel-norm err/1e-2"
    _report(f"{name} {op} {kind} {ratio:.4f} elements {out.numel()}")
    # bit-for-bit determinism
    out2 = _run(cg, op, pb, xd, wd, dyd)
    assert torch.equal(out.view(torch.int16 if out.dtype == torch.bfloat16 else torch.int32),
                       out2.view(torch.int16 if out.dtype == torch.bfloat16 else torch.int32))


# ------------------------------------------------------------------ the plain C entry points
# The binding goes through the extended entry points; these call conv2d_fwd, conv2d_bwd_data and
# conv2d_bwd_filter themselves (the thirteen descriptor integers, dtype, device pointers, the
# workspace and the stream), as a C caller would.
@pytest.mark.parametrize("name", ["tiny", "resnet3x3"])
def test_plain_entry_points(cg, name):
    import ctypes
    lib = cg.load_library()
    wl = W.WORKLOADS[name]
    pb = wl.problem
    x, w, dy = W.make_inputs(wl)
    xd, wd, dyd = x.to(DEV), w.to(DEV), dy.to(DEV)
    dt = 0 if pb.dtype == "f32" else 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    vp = lambda t: ctypes.c_void_p(t.data_ptr())
    for op, fn, a, b, shape in ((0, lib.conv2d_fwd, xd, wd, pb.y_shape),
                                (1, lib.conv2d_bwd_data, dyd, wd, pb.x_shape),
                                (2, lib.conv2d_bwd_filter, xd, dyd, pb.w_shape)):
        size = ctypes.c_size_t(0)
        assert lib.conv2d_workspace_size(op, *pb.dims(), dt, ctypes.byref(size)) == 0
        ws = torch.empty(max(size.value, 16), dtype=torch.uint8, device=DEV)
        out = _poisoned(shape, x.dtype)
        rc = fn(*pb.dims(), dt, vp(a), vp(b), vp(out), vp(ws), ctypes.c_size_t(size.value), stream)
        assert rc == 0, f"{name}/op {op}: {cg.conv2d_strerror(rc)}"
        assert lib.conv2d_device_status(stream) == 0
        opn = OPS[op]
        ra, rb = _operands(opn, x, w, dy)
        ratio = _check(opn, pb, out.double().cpu().numpy(), _oracle_full(opn, pb, x, w, dy), ra, rb,
                       f"plain/{name}/{opn}")
        _report(f"plain-entry {name} {opn} max|err|/tol {ratio:.4f}")


# ------------------------------------------------------------------ ragged small shapes
SMALL = [
    # N, C, H, W, K, R, S, ph, pw, sh, sw
    (1, 1, 5, 5, 1, 3, 3, 1, 1, 1, 1),
    (2, 3, 7, 9, 5, 3, 2, 1, 0, 1, 1),       # R != S, H != W
    (1, 5, 14, 7, 3, 3, 3, 1, 1, 2, 2),      # W*4 bytes not 16-byte aligned
    (2, 4, 9, 11, 6, 5, 3, 2, 1, 3, 2),      # stride 3 x 2, trailing rows uncovered
    (1, 2, 6, 13, 2, 6, 13, 0, 0, 1, 1),     # H == R, W == S
    (3, 7, 10, 10, 9, 1, 1, 0, 0, 1, 1),     # 1x1
    (1, 3, 12, 12, 16, 7, 7, 3, 3, 2, 2),    # stem-like
    (2, 8, 8, 8, 4, 4, 4, 1, 1, 2, 2),       # deconvolution-like 4x4 / 2
    (1, 33, 9, 9, 40, 3, 3, 1, 1, 1, 1),     # channel counts off every chunk size
    (1, 17, 6, 6, 300, 3, 3, 1, 1, 1, 1),    # K > 256: several N tiles
    (2, 70, 11, 5, 130, 2, 2, 0, 1, 1, 2),
    (2, 3, 20, 20, 8, 5, 5, 0, 0, 5, 5),     # stride 5 x 5: 25 phase planes, non-overlapping windows
    (1, 6, 27, 26, 5, 3, 4, 1, 2, 6, 5),     # stride 6 x 5: 30 planes
    (1, 1, 4, 4, 1, 1, 1, 0, 0, 3, 3),       # 1x1 stride 3: backward-data phases without taps
    (4, 12, 20, 20, 24, 3, 3, 0, 0, 1, 1),   # no padding
    (1, 9, 31, 17, 11, 5, 5, 2, 2, 1, 1),
    (2, 300, 5, 5, 20, 3, 3, 1, 1, 1, 1),    # C > 256: several channel blocks
    # backward-filter row-tap sharing (unit stride, C >= 32, aligned rows)
    (2, 64, 16, 16, 64, 3, 3, 1, 1, 1, 1),   # 3 filter rows per unit
    (1, 40, 16, 16, 48, 5, 3, 2, 1, 1, 1),   # row blocks of 4 + 1, a partial channel group
    (1, 32, 16, 16, 150, 3, 3, 1, 1, 1, 1),  # wide k tile: row blocks of 2 + 1
    (1, 32, 6, 48, 64, 3, 3, 1, 1, 1, 1),    # wide rows (bf16 shares rows too)
    (2, 48, 10, 16, 20, 3, 5, 1, 2, 1, 1),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", SMALL)
@pytest.mark.parametrize("op", OPS)
def test_small_parity(cg, case, op, dtype):
    N, C, H, Wd, K, R, S, ph, pw, sh, sw = case
    pb = W.Conv2dProblem(N, C, H, Wd, K, R, S, ph, pw, sh, sw, dtype)
    x, w, dy = W.random_problem_inputs(pb, 7000 + SMALL.index(case))
    out = _run(cg, op, pb, x.to(DEV), w.to(DEV), dy.to(DEV))
    assert not torch.isnan(out).any().item()
    ref = _oracle_full(op, pb, x, w, dy)
    a, b = _operands(op, x, w, dy)
    _check(op, pb, out.double().cpu().numpy(), ref, a, b, f"{case}/{op}/{dtype}")


# ------------------------------------------------------------------ wide bf16 layers
# bf16 layers with 256 or more destination channels, whose filter slice is most of a stage (tiles
# of 256 destination channels, tap-pair stages): an odd m-tile count, a ragged second
# destination-channel tile, stride phases on both ops.
WIDE_CASES = [
    # N, C, H, W, K, R, S, ph, pw, sh, sw
    (4, 16, 16, 16, 256, 4, 4, 1, 1, 2, 2),   # forward, 3 m-tiles
    (4, 256, 16, 16, 16, 4, 4, 1, 1, 2, 2),   # backward-data, 4 output phases
    (3, 8, 20, 18, 272, 3, 3, 1, 1, 1, 1),    # forward, K = 272: a ragged second tile
    (6, 272, 14, 14, 8, 4, 4, 1, 1, 2, 2),    # backward-data, C = 272
]


@pytest.mark.parametrize("case", WIDE_CASES)
@pytest.mark.parametrize("op", ["fwd", "bwd_data"])
def test_wide_bf16_parity(cg, case, op):
    N, C, H, Wd, K, R, S, ph, pw, sh, sw = case
    pb = W.Conv2dProblem(N, C, H, Wd, K, R, S, ph, pw, sh, sw, "bf16")
    x, w, dy = W.random_problem_inputs(pb, 7600 + WIDE_CASES.index(case))
    out = _run(cg, op, pb, x.to(DEV), w.to(DEV), dy.to(DEV))
    assert not torch.isnan(out).any().item()
    ref = _oracle_full(op, pb, x, w, dy)
    a, b = _operands(op, x, w, dy)
    _check(op, pb, out.double().cpu().numpy(), ref, a, b, f"wide {case}/{op}")


@pytest.mark.parametrize("op", ["fwd", "bwd_data"])
def test_bf16_strided_two_half_tiles(cg, op):
    """A bf16 stride-2 layer large enough for 256-row tiles (two accumulator halves), whose
    staged rows (312 per plane) exceed one copy's box: the forward stages its four stride-phase
    planes with one copy per plane and box of rows."""
    pb = W.Conv2dProblem(64, 16, 64, 64, 64, 3, 3, 1, 1, 2, 2, "bf16")
    x, w, dy = W.random_problem_inputs(pb, 7900)
    out = _run(cg, op, pb, x.to(DEV), w.to(DEV), dy.to(DEV))
    assert not torch.isnan(out).any().item()
    a, b = _operands(op, x, w, dy)
    _check(op, pb, out.double().cpu().numpy(), _oracle_full(op, pb, x, w, dy), a, b, f"two-half {op}")


@pytest.mark.parametrize("case", WIDE_CASES[:2])
def test_wide_bf16_fused_epilogue(cg, case):
    """The fused epilogue (bias and add-to) on the wide bf16 layers, both ops."""
    N, C, H, Wd, K, R, S, ph, pw, sh, sw = case
    pb = W.Conv2dProblem(N, C, H, Wd, K, R, S, ph, pw, sh, sw, "bf16")
    x, w, dy = W.random_problem_inputs(pb, 7700 + WIDE_CASES.index(case))
    g = torch.Generator().manual_seed(7800 + WIDE_CASES.index(case))
    bk = torch.randn(K, generator=g).to(torch.bfloat16)
    bc = torch.randn(C, generator=g).to(torch.bfloat16)
    y0 = torch.randn(pb.y_shape, generator=g).to(torch.bfloat16)
    dx0 = torch.randn(pb.x_shape, generator=g).to(torch.bfloat16)
    pad, st = (ph, pw), (sh, sw)
    amax = lambda t: float(t.abs().max())
    y = y0.to(DEV)
    cg.conv2d_fwd(x.to(DEV), w.to(DEV), pad, st, out=y, bias=bk.to(DEV), beta=1.0)
    dx = dx0.to(DEV)
    cg.conv2d_bwd_data(dy.to(DEV), w.to(DEV), (H, Wd), pad, st, out=dx, bias=bc.to(DEV), beta=0.5)
    cg.conv2d_device_status()
    _check_plain(pb, y.double().cpu().numpy(), oracle.conv2d_fwd_ex(x, w, bk, 1.0, y0, pad, st),
                 amax(x) * amax(w), C * R * S, f"wide {case}/fwd_ex")
    _check_plain(pb, dx.double().cpu().numpy(), oracle.conv2d_bwd_data_ex(dy, w, (H, Wd), bc, 0.5, dx0, pad, st),
                 amax(dy) * amax(w), K * R * S, f"wide {case}/bwd_data_ex")


def test_deconv_alias_matches_oracle_scatter(cg):
    """deconv2d_fwd (= backward-data with the weight read as (in, out, R, S)) against
    the oracle's independent scatter-form transposed convolution."""
    g = torch.Generator().manual_seed(99)
    inp = torch.randn(2, 12, 5, 5, generator=g)
    wt = torch.randn(12, 7, 4, 4, generator=g)
    out = cg.deconv2d_fwd(inp.to(DEV), wt.to(DEV), (10, 10), 1, 2)
    cg.conv2d_device_status()
    ref = oracle.deconv2d_fwd_scatter(inp, wt, (10, 10), 1, 2)
    tol = 2e-3 * math.sqrt(12 * 16 / 4) * float(inp.abs().max()) * float(wt.abs().max())
    assert float(np.abs(out.double().cpu().numpy() - ref).max()) <= tol


def test_stream_argument_is_honoured(cg):
    pb = W.WORKLOADS["tiny"].problem
    x, w, dy = W.make_inputs(W.WORKLOADS["tiny"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = cg.conv2d_fwd(x.to(DEV), w.to(DEV), 1, 1, stream=s)
    s.synchronize()
    ref = oracle.conv2d_fwd(x, w, 1, 1)
    assert float(np.abs(y.double().cpu().numpy() - ref).max()) <= 2e-3 * math.sqrt(27)


def test_timeout_flag_clear_after_normal_runs(cg):
    assert cg.conv2d_device_status() == 0


# ------------------------------------------------------------------ fused epilogues
# bias + beta * old on every output, bias gradients over dy (per k) and x (per c).
EPI_CASES = [
    (2, 3, 7, 9, 5, 3, 2, 1, 0, 1, 1),
    (1, 33, 9, 9, 40, 3, 3, 1, 1, 1, 1),
    (2, 64, 16, 16, 64, 3, 3, 1, 1, 1, 1),   # backward-filter row-tap sharing
    (2, 8, 8, 8, 4, 4, 4, 1, 1, 2, 2),
]


def _check_plain(pb, got, ref, scale, length, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if pb.dtype == "f32":
        tol = 2e-3 * math.sqrt(length) * scale
        err = float(np.abs(got - ref).max(initial=0.0))
        assert err <= tol, f"{what}: max|err| {err:.3e} > {tol:.3e}"
    else:
        den = float(np.linalg.norm(ref))
        rel = float(np.linalg.norm(got - ref)) / den if den > 0 else float(np.linalg.norm(got))
        assert rel <= 1e-2, f"{what}: relative-to-norm error {rel:.3e} > 1e-2"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", EPI_CASES)
def test_fused_epilogue_parity(cg, case, dtype):
    N, C, H, Wd, K, R, S, ph, pw, sh, sw = case
    pb = W.Conv2dProblem(N, C, H, Wd, K, R, S, ph, pw, sh, sw, dtype)
    x, w, dy = W.random_problem_inputs(pb, 9100 + EPI_CASES.index(case))
    tdt = x.dtype
    g = torch.Generator().manual_seed(9200 + EPI_CASES.index(case))
    bk = torch.randn(K, generator=g).to(tdt)
    bc = torch.randn(C, generator=g).to(tdt)
    y0 = torch.randn(pb.y_shape, generator=g).to(tdt)
    dx0 = torch.randn(pb.x_shape, generator=g).to(tdt)
    dw0 = torch.randn(pb.w_shape, generator=g).to(tdt)
    dbk0 = torch.randn(K, generator=g).to(tdt)
    dbc0 = torch.randn(C, generator=g).to(tdt)
    pad, st = (ph, pw), (sh, sw)
    xd, wd, dyd = x.to(DEV), w.to(DEV), dy.to(DEV)
    amax = lambda t: float(t.abs().max())

    y = y0.to(DEV)
    cg.conv2d_fwd(xd, wd, pad, st, out=y, bias=bk.to(DEV), beta=1.0)
    dx = dx0.to(DEV)
    cg.conv2d_bwd_data(dyd, wd, (H, Wd), pad, st, out=dx, bias=bc.to(DEV), beta=0.5)
    dw, dbk, dbc = dw0.to(DEV), dbk0.to(DEV), dbc0.to(DEV)
    cg.conv2d_bwd_filter(xd, dyd, (R, S), pad, st, out=dw, beta=1.0, db_k=dbk, db_c=dbc)
    cg.conv2d_device_status()

    _check_plain(pb, y.double().cpu().numpy(), oracle.conv2d_fwd_ex(x, w, bk, 1.0, y0, pad, st),
                 amax(x) * amax(w), C * R * S, f"{case}/fwd_ex/{dtype}")
    _check_plain(pb, dx.double().cpu().numpy(), oracle.conv2d_bwd_data_ex(dy, w, (H, Wd), bc, 0.5, dx0, pad, st),
                 amax(dy) * amax(w), K * R * S, f"{case}/bwd_data_ex/{dtype}")
    _check_plain(pb, dw.double().cpu().numpy(), oracle.conv2d_bwd_filter_ex(x, dy, (R, S), 1.0, dw0, pad, st),
                 amax(x) * amax(dy), N * pb.P * pb.Q, f"{case}/bwd_filter_ex/{dtype}")
    _check_plain(pb, dbk.double().cpu().numpy(), oracle.channel_sum(dy, 1.0, dbk0),
                 amax(dy), N * pb.P * pb.Q, f"{case}/db_k/{dtype}")
    _check_plain(pb, dbc.double().cpu().numpy(), oracle.channel_sum(x, 1.0, dbc0),
                 amax(x), N * H * Wd, f"{case}/db_c/{dtype}")


def test_bias_gradient_resnet_workload(cg):
    """Bias gradients at the full ResNet 3x3 size (every channel, exact fp64 reference)."""
    wl = W.WORKLOADS["resnet3x3"]
    pb = wl.problem
    x, w, dy = W.make_inputs(wl)
    K, C = pb.K, pb.C
    dbk = _poisoned((K,), x.dtype)
    dbc = _poisoned((C,), x.dtype)
    dw = _poisoned(pb.w_shape, x.dtype)
    cg.conv2d_bwd_filter(x.to(DEV), dy.to(DEV), (pb.R, pb.S), (pb.pad_h, pb.pad_w), (pb.stride_h, pb.stride_w),
                         out=dw, db_k=dbk, db_c=dbc)
    cg.conv2d_device_status()
    for got, t, length in ((dbk, dy, pb.N * pb.P * pb.Q), (dbc, x, pb.N * pb.H * pb.W)):
        ref = oracle.channel_sum(t)
        err = float(np.abs(got.double().cpu().numpy() - ref).max())
        assert err <= 2e-3 * math.sqrt(length) * float(t.abs().max())


# ------------------------------------------------------------------ convolution mode, 1-D
FLIP_CASES = [
    (2, 3, 7, 9, 5, 3, 2, 1, 0, 1, 1),
    (1, 5, 14, 7, 3, 3, 3, 1, 1, 2, 2),
    (2, 64, 16, 16, 64, 3, 3, 1, 1, 1, 1),   # backward-filter row-tap sharing
    (2, 40, 23, 19, 24, 3, 3, 1, 1, 3, 2),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", FLIP_CASES)
def test_convolution_mode_parity(cg, case, dtype):
    N, C, H, Wd, K, R, S, ph, pw, sh, sw = case
    pb = W.Conv2dProblem(N, C, H, Wd, K, R, S, ph, pw, sh, sw, dtype)
    x, w, dy = W.random_problem_inputs(pb, 9300 + FLIP_CASES.index(case))
    pad, st = (ph, pw), (sh, sw)
    xd, wd, dyd = x.to(DEV), w.to(DEV), dy.to(DEV)
    y = _poisoned(pb.y_shape, x.dtype)
    cg.conv2d_fwd(xd, wd, pad, st, out=y, flip=True)
    dx = _poisoned(pb.x_shape, x.dtype)
    cg.conv2d_bwd_data(dyd, wd, (H, Wd), pad, st, out=dx, flip=True)
    dw = _poisoned(pb.w_shape, x.dtype)
    cg.conv2d_bwd_filter(xd, dyd, (R, S), pad, st, out=dw, flip=True)
    cg.conv2d_device_status()
    for op, got, ref in (("fwd", y, oracle.conv2d_fwd_ex(x, w, None, 0.0, None, pad, st, flip=True)),
                         ("bwd_data", dx, oracle.conv2d_bwd_data_ex(dy, w, (H, Wd), None, 0.0, None, pad, st, flip=True)),
                         ("bwd_filter", dw, oracle.conv2d_bwd_filter_ex(x, dy, (R, S), 0.0, None, pad, st, flip=True))):
        a, b = _operands(op, x, w, dy)
        _check(op, pb, got.double().cpu().numpy(), ref, a, b, f"{case}/{op}/flip/{dtype}")


@pytest.mark.parametrize("flip", [False, True])
def test_conv1d_wrappers(cg, flip):
    """conv1d_* = the 2-D ops with H = R = 1, checked against the oracle on (N, C, 1, W)."""
    g = torch.Generator().manual_seed(9400 + int(flip))
    N, C, Wd, K, S, pad, stride = 3, 6, 29, 5, 4, 2, 2
    Q = (Wd + 2 * pad - S) // stride + 1
    x = torch.randn(N, C, Wd, generator=g)
    w = torch.randn(K, C, S, generator=g)
    dy = torch.randn(N, K, Q, generator=g)
    y = cg.conv1d_fwd(x.to(DEV), w.to(DEV), pad, stride, flip=flip)
    dx = cg.conv1d_bwd_data(dy.to(DEV), w.to(DEV), Wd, pad, stride, flip=flip)
    dw = cg.conv1d_bwd_filter(x.to(DEV), dy.to(DEV), S, pad, stride, flip=flip)
    cg.conv2d_device_status()
    x4, w4, dy4 = x.unsqueeze(2), w.unsqueeze(2), dy.unsqueeze(2)
    refs = (oracle.conv2d_fwd_ex(x4, w4, None, 0.0, None, (0, pad), (1, stride), flip=flip)[:, :, 0],
            oracle.conv2d_bwd_data_ex(dy4, w4, (1, Wd), None, 0.0, None, (0, pad), (1, stride), flip=flip)[:, :, 0],
            oracle.conv2d_bwd_filter_ex(x4, dy4, (1, S), 0.0, None, (0, pad), (1, stride), flip=flip)[:, :, 0])
    lens = (C * S, K * S, N * Q)
    amax = [float(t.abs().max()) for t in (x, w, dy)]
    scales = (amax[0] * amax[1], amax[2] * amax[1], amax[0] * amax[2])
    for got, ref, L, sc in zip((y, dx, dw), refs, lens, scales):
        assert tuple(got.shape) == ref.shape
        err = float(np.abs(got.double().cpu().numpy() - ref).max())
        assert err <= 2e-3 * math.sqrt(L) * sc


# ------------------------------------------------------------------ dilation
DIL_GPU_CASES = [
    ((2, 8, 12, 13, 6, 3, 3, 2, 2, 1, 1), (2, 2)),
    ((1, 5, 20, 17, 7, 3, 2, 2, 1, 2, 1), (2, 3)),
    ((2, 64, 16, 16, 64, 3, 3, 2, 2, 1, 1), (2, 2)),    # copy-engine staging, no row-tap sharing
    ((1, 33, 15, 16, 40, 2, 3, 1, 2, 1, 2), (3, 2)),
    ((2, 3, 21, 21, 16, 3, 3, 3, 3, 2, 2), (3, 3)),     # few channels, stride 2
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case,dil", DIL_GPU_CASES)
def test_dilation_parity(cg, case, dil, dtype):
    N, C, H, Wd, K, R, S, ph, pw, sh, sw = case
    dh, dw_ = dil
    P = (H + 2 * ph - dh * (R - 1) - 1) // sh + 1
    Q = (Wd + 2 * pw - dw_ * (S - 1) - 1) // sw + 1
    g = torch.Generator().manual_seed(9500 + DIL_GPU_CASES.index((case, dil)))
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    x = torch.randn(N, C, H, Wd, generator=g).to(tdt)
    w = torch.randn(K, C, R, S, generator=g).to(tdt)
    dy = torch.randn(N, K, P, Q, generator=g).to(tdt)
    pad, st = (ph, pw), (sh, sw)
    flip = DIL_GPU_CASES.index((case, dil)) % 2 == 1
    xd, wd, dyd = x.to(DEV), w.to(DEV), dy.to(DEV)
    y = _poisoned((N, K, P, Q), tdt)
    cg.conv2d_fwd(xd, wd, pad, st, out=y, dilation=dil, flip=flip)
    dx = _poisoned((N, C, H, Wd), tdt)
    cg.conv2d_bwd_data(dyd, wd, (H, Wd), pad, st, out=dx, dilation=dil, flip=flip)
    dwt = _poisoned((K, C, R, S), tdt)
    cg.conv2d_bwd_filter(xd, dyd, (R, S), pad, st, out=dwt, dilation=dil, flip=flip)
    cg.conv2d_device_status()
    amax = lambda t: float(t.abs().max())
    checks = (("fwd", y, oracle.conv2d_fwd_ex(x, w, None, 0.0, None, pad, st, flip, dil), amax(x) * amax(w), C * R * S),
              ("bwd_data", dx, oracle.conv2d_bwd_data_ex(dy, w, (H, Wd), None, 0.0, None, pad, st, flip, dil),
               amax(dy) * amax(w), K * R * S),
              ("bwd_filter", dwt, oracle.conv2d_bwd_filter_ex(x, dy, (R, S), 0.0, None, pad, st, flip, dil),
               amax(x) * amax(dy), N * P * Q))
    for op, got, ref, scale, L in checks:
        got = got.double().cpu().numpy()
        assert np.all(np.isfinite(got)), f"{case}/{dil}/{op}: unwritten element"
        if dtype == "f32":
            err = float(np.abs(got - ref).max())
            assert err <= 2e-3 * math.sqrt(L) * scale, f"{case}/{dil}/{op}: {err:.3e}"
        else:
            den = float(np.linalg.norm(ref))
            rel = float(np.linalg.norm(got - ref)) / den if den > 0 else float(np.linalg.norm(got))
            assert rel <= 1e-2, f"{case}/{dil}/{op}: {rel:.3e}"


# ------------------------------------------------------------------ groups
GROUP_GPU_CASES = [
    ((2, 6, 9, 10, 9, 3, 3, 1, 1, 1, 1), 3, (1, 1), False),
    ((1, 16, 12, 12, 16, 3, 3, 1, 1, 1, 1), 16, (1, 1), True),    # depthwise
    ((2, 64, 16, 16, 64, 3, 3, 1, 1, 1, 1), 2, (1, 1), False),    # copy-engine staging per group
    ((2, 8, 13, 11, 6, 3, 3, 2, 2, 1, 2), 2, (2, 1), True),
    ((2, 36, 14, 15, 20, 3, 3, 1, 1, 2, 2), 2, (1, 1), False),  # two groups of 18: chunks straddle the groups
    ((2, 32, 12, 13, 48, 3, 3, 1, 1, 1, 1), 4, (1, 1), True),   # four groups of 8 -> 12
    ((2, 24, 15, 13, 24, 5, 5, 2, 2, 2, 2), 24, (1, 1), False),  # depthwise 5x5, stride 2
    ((2, 8, 12, 12, 16, 3, 3, 2, 2, 1, 1), 8, (2, 2), False),    # depthwise, 2 outputs per channel, dilation 2
    ((1, 5, 7, 9, 10, 3, 2, 1, 0, 2, 1), 5, (1, 1), True),       # depthwise x2, R != S, stride 2 x 1
    ((2, 4, 1, 20000, 4, 1, 5, 0, 2, 1, 1), 4, (1, 1), False),   # depthwise 1-D, rows too wide to stage
    ((2, 6, 20, 18, 6, 7, 7, 3, 3, 1, 1), 6, (1, 1), True),      # depthwise 7x7
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case,groups,dil,flip", GROUP_GPU_CASES)
def test_groups_parity(cg, case, groups, dil, flip, dtype):
    N, C, H, Wd, K, R, S, ph, pw, sh, sw = case
    dh, dw_ = dil
    P = (H + 2 * ph - dh * (R - 1) - 1) // sh + 1
    Q = (Wd + 2 * pw - dw_ * (S - 1) - 1) // sw + 1
    idx = [c[0] for c in GROUP_GPU_CASES].index(case)
    g = torch.Generator().manual_seed(9600 + idx)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    x = torch.randn(N, C, H, Wd, generator=g).to(tdt)
    w = torch.randn(K, C // groups, R, S, generator=g).to(tdt)
    dy = torch.randn(N, K, P, Q, generator=g).to(tdt)
    bk = torch.randn(K, generator=g).to(tdt)
    y0 = torch.randn(N, K, P, Q, generator=g).to(tdt)
    pad, st = (ph, pw), (sh, sw)
    xd, wd, dyd = x.to(DEV), w.to(DEV), dy.to(DEV)
    y = y0.to(DEV)
    cg.conv2d_fwd(xd, wd, pad, st, out=y, bias=bk.to(DEV), beta=1.0, dilation=dil, groups=groups, flip=flip)
    dx = _poisoned((N, C, H, Wd), tdt)
    cg.conv2d_bwd_data(dyd, wd, (H, Wd), pad, st, out=dx, dilation=dil, groups=groups, flip=flip)
    dwt = _poisoned((K, C // groups, R, S), tdt)
    dbk = _poisoned((K,), tdt)
    cg.conv2d_bwd_filter(xd, dyd, (R, S), pad, st, out=dwt, dilation=dil, groups=groups, flip=flip, db_k=dbk)
    cg.conv2d_device_status()
    amax = lambda t: float(t.abs().max())
    checks = (("fwd", y, oracle.conv2d_fwd_ex(x, w, bk, 1.0, y0, pad, st, flip, dil, groups), amax(x) * amax(w),
               (C // groups) * R * S),
              ("bwd_data", dx, oracle.conv2d_bwd_data_ex(dy, w, (H, Wd), None, 0.0, None, pad, st, flip, dil, groups),
               amax(dy) * amax(w), (K // groups) * R * S),
              ("bwd_filter", dwt, oracle.conv2d_bwd_filter_ex(x, dy, (R, S), 0.0, None, pad, st, flip, dil, groups),
               amax(x) * amax(dy), N * P * Q),
              ("db_k", dbk, oracle.channel_sum(dy), amax(dy), N * P * Q))
    for op, got, ref, scale, L in checks:
        got = got.double().cpu().numpy()
        assert np.all(np.isfinite(got)), f"{case}/g{groups}/{op}: unwritten element"
        if dtype == "f32":
            err = float(np.abs(got - ref).max())
            assert err <= 2e-3 * math.sqrt(L) * scale, f"{case}/g{groups}/{op}: {err:.3e}"
        else:
            den = float(np.linalg.norm(ref))
            rel = float(np.linalg.norm(got - ref)) / den if den > 0 else float(np.linalg.norm(got))
            assert rel <= 1e-2, f"{case}/g{groups}/{op}: {rel:.3e}"


# Large filters whose filter slices do not fit the tap GEMM's shared memory in one pass: the
# taps run in contiguous ranges, the first pass with the caller's bias and beta, the later
# ones adding on.  The comment gives the passes the planner makes (forward, backward-data).
PASS_CASES = [
    ((1, 16, 40, 40, 16, 16, 16, 7, 7, 1, 1), "f32"),   # 1, 1 (tap pairs: 256 taps in one pass)
    ((1, 32, 40, 40, 32, 16, 16, 7, 7, 1, 1), "f32"),   # 2, 2
    ((1, 64, 30, 30, 64, 13, 13, 6, 6, 1, 1), "f32"),   # 2, 2
    ((2, 24, 40, 40, 20, 16, 16, 7, 7, 2, 2), "bf16"),  # 2, 1
    ((1, 40, 40, 40, 96, 15, 15, 7, 7, 1, 1), "bf16"),  # 4, 2
    ((1, 64, 4, 300, 64, 1, 256, 0, 3, 1, 1), "f32"),   # 3, 3
    ((1, 4, 40, 40, 8, 17, 17, 8, 8, 1, 1), "f32"),     # 2, 2 (289 taps: more than one pass holds)
    ((1, 8, 36, 36, 16, 17, 17, 8, 8, 1, 1), "bf16"),   # 2, 2
]


@pytest.mark.parametrize("epi", [False, True])
@pytest.mark.parametrize("case,dtype", PASS_CASES)
def test_tap_passes_parity(cg, case, dtype, epi):
    N, C, H, Wd, K, R, S, ph, pw, sh, sw = case
    pb = W.Conv2dProblem(N, C, H, Wd, K, R, S, ph, pw, sh, sw, dtype)
    seed = 9500 + 2 * PASS_CASES.index((case, dtype)) + int(epi)
    x, w, dy = W.random_problem_inputs(pb, seed)
    tdt = x.dtype
    g = torch.Generator().manual_seed(seed)
    bk = torch.randn(K, generator=g).to(tdt) if epi else None
    bc = torch.randn(C, generator=g).to(tdt) if epi else None
    y0 = torch.randn(pb.y_shape, generator=g).to(tdt)
    dx0 = torch.randn(pb.x_shape, generator=g).to(tdt)
    beta_f, beta_d = (1.0, 0.5) if epi else (0.0, 0.0)
    pad, st = (ph, pw), (sh, sw)
    xd, wd, dyd = x.to(DEV), w.to(DEV), dy.to(DEV)
    amax = lambda t: float(t.abs().max())
    y = y0.to(DEV) if epi else _poisoned(pb.y_shape, tdt)
    cg.conv2d_fwd(xd, wd, pad, st, out=y, bias=bk.to(DEV) if epi else None, beta=beta_f)
    dx = dx0.to(DEV) if epi else _poisoned(pb.x_shape, tdt)
    cg.conv2d_bwd_data(dyd, wd, (H, Wd), pad, st, out=dx, bias=bc.to(DEV) if epi else None, beta=beta_d)
    cg.conv2d_device_status()
    _check_plain(pb, y.double().cpu().numpy(), oracle.conv2d_fwd_ex(x, w, bk, beta_f, y0, pad, st),
                 amax(x) * amax(w), C * R * S, f"{case}/fwd/{dtype}/epi={epi}")
    _check_plain(pb, dx.double().cpu().numpy(), oracle.conv2d_bwd_data_ex(dy, w, (H, Wd), bc, beta_d, dx0, pad, st),
                 amax(dy) * amax(w), K * R * S, f"{case}/bwd_data/{dtype}/epi={epi}")


# Strided backward-filter (dilation 1) runs as stride phases where that stages less than the
# problem as a whole: x copied once into unit-stride planes, one stride-1 pass per phase whose
# reduce places its taps in the filter.  Every case below takes the phases in both dtypes:
# groups, 4x4 stride 2, stride 3 with 2x2 taps (phases without taps), unequal strides, odd
# extents; each with convolution mode, beta and the bias gradient.
PHASE_CASES = [
    ((2, 256, 14, 14, 128, 3, 3, 1, 1, 2, 2), 2),
    ((1, 192, 20, 16, 160, 4, 4, 1, 1, 2, 2), 2),
    ((1, 128, 24, 24, 64, 2, 2, 0, 0, 3, 3), 1),
    ((1, 128, 23, 22, 96, 2, 3, 0, 1, 3, 2), 1),
    ((2, 128, 15, 14, 64, 3, 3, 1, 1, 2, 2), 1),
    ((1, 96, 25, 23, 64, 3, 3, 1, 1, 3, 3), 1),
    ((1, 64, 22, 21, 32, 5, 3, 2, 1, 2, 3), 1),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("flip", [False, True])
@pytest.mark.parametrize("case,groups", PHASE_CASES)
def test_stride_phase_bwd_filter_parity(cg, case, groups, flip, dtype):
    N, C, H, Wd, K, R, S, ph, pw, sh, sw = case
    pb = W.Conv2dProblem(N, C, H, Wd, K, R, S, ph, pw, sh, sw, dtype)
    seed = 9700 + 4 * PHASE_CASES.index((case, groups)) + 2 * int(flip) + int(dtype == "bf16")
    x, _, dy = W.random_problem_inputs(pb, seed)
    tdt = x.dtype
    g = torch.Generator().manual_seed(seed)
    dw0 = torch.randn((K, C // groups, R, S), generator=g).to(tdt)
    dbk0 = torch.randn(K, generator=g).to(tdt)
    pad, st = (ph, pw), (sh, sw)
    dw, dbk = dw0.to(DEV), dbk0.to(DEV)
    cg.conv2d_bwd_filter(x.to(DEV), dy.to(DEV), (R, S), pad, st, out=dw, beta=0.5, db_k=dbk, flip=flip,
                         groups=groups)
    cg.conv2d_device_status()
    amax = lambda t: float(t.abs().max())
    ref = oracle.conv2d_bwd_filter_ex(x, dy, (R, S), 0.5, dw0, pad, st, flip=flip, groups=groups)
    _check_plain(pb, dw.double().cpu().numpy(), ref, amax(x) * amax(dy), N * pb.P * pb.Q,
                 f"{case}/g{groups}/flip={flip}/{dtype}")
    _check_plain(pb, dbk.double().cpu().numpy(), oracle.channel_sum(dy, 0.5, dbk0), amax(dy), N * pb.P * pb.Q,
                 f"{case}/db_k/{dtype}")


# 3-D (NCDHW): every element of the three ops against the fp64 3-D oracle.  Each case is
# N, C, (D, H, W), K, (T, R, S), pads, strides, dilations, groups.
CASES_3D = [
    (2, 3, (5, 6, 7), 4, (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), 1),
    (1, 8, (7, 9, 8), 6, (3, 3, 2), (1, 1, 0), (2, 2, 1), (1, 1, 1), 1),     # depth and row stride 2
    (2, 4, (6, 8, 8), 4, (2, 3, 3), (0, 2, 1), (1, 1, 2), (2, 2, 1), 2),     # depth dilation 2, groups 2
    (1, 16, (4, 10, 10), 24, (3, 1, 1), (1, 0, 0), (1, 1, 1), (1, 1, 1), 1),  # depth-only filter
    (1, 5, (9, 5, 6), 7, (4, 2, 3), (2, 1, 1), (3, 1, 1), (1, 1, 1), 1),     # depth stride 3, uncovered tail
]


def _red_len_3d(op, N, C, K, T, R, S, Z, P, Q, st, groups):
    if op == "fwd":
        return (C // groups) * T * R * S
    if op == "bwd_data":
        return (K // groups) * math.ceil(T / st[0]) * math.ceil(R / st[1]) * math.ceil(S / st[2])
    return N * Z * P * Q


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("op", ["fwd", "bwd_data", "bwd_filter"])
@pytest.mark.parametrize("case", CASES_3D)
def test_conv3d_parity(cg, case, op, dtype):
    N, C, dhw, K, trs, pad, st, dil, groups = case
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    g = torch.Generator().manual_seed(9700 + CASES_3D.index(case))
    x = (torch.rand((N, C, *dhw), generator=g) * 2 - 1).to(tdt)
    w = (torch.rand((K, C // groups, *trs), generator=g) * 2 - 1).to(tdt)
    zpq = tuple((i + 2 * p - (d * (k - 1) + 1)) // s + 1 for i, p, k, s, d in zip(dhw, pad, trs, st, dil))
    dy = (torch.rand((N, K, *zpq), generator=g) * 2 - 1).to(tdt)
    if op == "fwd":
        out = cg.conv3d_fwd(x.to(DEV), w.to(DEV), pad, st, dil, groups)
        ref = oracle.conv3d_fwd(x, w, pad, st, dil, groups)
        a, b = x, w
    elif op == "bwd_data":
        out = cg.conv3d_bwd_data(dy.to(DEV), w.to(DEV), dhw, pad, st, dil, groups)
        ref = oracle.conv3d_bwd_data(dy, w, dhw, pad, st, dil, groups)
        a, b = dy, w
    else:
        out = cg.conv3d_bwd_filter(x.to(DEV), dy.to(DEV), trs, pad, st, dil, groups)
        ref = oracle.conv3d_bwd_filter(x, dy, trs, pad, st, dil, groups)
        a, b = x, dy
    cg.conv2d_device_status()
    pb = W.Conv2dProblem(1, 1, 1, 1, 1, 1, 1, dtype=dtype)  # carries the dtype for the check
    length = _red_len_3d(op, N, C, K, *trs, *zpq, st, groups)
    _check_plain(pb, out.double().cpu().numpy(), ref, float(a.abs().max()) * float(b.abs().max()), length,
                 f"3-D {case}/{op}/{dtype}")



# Both gradients in one call (conv2d_bwd): every element of dx and dw against the full oracle,
# and bit for bit equal to the two single operations (the same plans; with bf16 the
# backward-data GEMM reads the backward-filter plan's dy pack).
@pytest.mark.parametrize("name", ["deconv", "resnet3x3", "tiny"])
def test_fused_backward_parity(cg, name):
    wl = W.WORKLOADS[name]
    pb = wl.problem
    x, w, dy = W.make_inputs(wl)
    xd, wd, dyd = x.to(DEV), w.to(DEV), dy.to(DEV)
    pad, st = (pb.pad_h, pb.pad_w), (pb.stride_h, pb.stride_w)
    dx, dw = cg.conv2d_bwd(xd, wd, dyd, pad, st)
    dx1 = cg.conv2d_bwd_data(dyd, wd, (pb.H, pb.W), pad, st)
    dw1 = cg.conv2d_bwd_filter(xd, dyd, (pb.R, pb.S), pad, st)
    cg.conv2d_device_status()
    assert torch.equal(dx, dx1) and torch.equal(dw, dw1), f"{name}: fused backward differs from the single ops"
    for op, out in (("bwd_data", dx), ("bwd_filter", dw)):
        ref = _oracle_cached(op, name, pb, x, w, dy)
        a, b = _operands(op, x, w, dy)
        _check(op, pb, out.double().cpu().numpy(), ref, a, b, f"{name}/fused {op}")


@pytest.mark.parametrize("case", [(2, 16, 12, 10, 24, 4, 4, 1, 1, 2, 2), (1, 8, 9, 11, 16, 3, 3, 1, 1, 2, 2)])
def test_fused_backward_small_bf16(cg, case):
    N, C, H, Wd, K, R, S, ph, pw, sh, sw = case
    pb = W.Conv2dProblem(N, C, H, Wd, K, R, S, ph, pw, sh, sw, "bf16")
    x, w, dy = W.random_problem_inputs(pb, 9800)
    dx, dw = cg.conv2d_bwd(x.to(DEV), w.to(DEV), dy.to(DEV), (ph, pw), (sh, sw))
    cg.conv2d_device_status()
    for op, out in (("bwd_data", dx), ("bwd_filter", dw)):
        ref = _oracle_full(op, pb, x, w, dy)
        a, b = _operands(op, x, w, dy)
        _check(op, pb, out.double().cpu().numpy(), ref, a, b, f"{case}/fused {op}")


# Backward-data with few input channels (C <= 8) runs the scatter-form kernel: Z = dy^T w on
# the tensor cores for 8 x 32 dy positions per tile, folded on chip into dx.  Cases: strides,
# dilations, halos up to the tile limits (5 dy rows, 7 dy columns), K not a multiple of the
# 32-channel block, groups, convolution mode, bias + add-to; image edges ragged in both axes.
C2I_CASES = [
    # (N, C, H, W, K, R, S, ph, pw, sh, sw), (dh, dw), groups, flip, epilogue
    ((1, 3, 37, 45, 16, 7, 7, 3, 3, 2, 2), (1, 1), 1, False, False),   # the stem's shape, small
    ((2, 1, 19, 70, 40, 3, 3, 1, 1, 1, 1), (1, 1), 1, True, False),
    ((1, 2, 23, 29, 8, 3, 3, 2, 2, 1, 1), (2, 2), 1, False, True),
    ((1, 4, 25, 22, 12, 5, 4, 1, 2, 3, 2), (1, 1), 1, True, True),
    ((3, 3, 12, 12, 33, 3, 3, 1, 1, 1, 1), (1, 1), 1, False, False),
    ((1, 4, 9, 40, 20, 1, 8, 0, 3, 1, 1), (1, 1), 1, False, True),
    ((1, 2, 18, 37, 7, 4, 4, 0, 1, 4, 4), (1, 1), 1, True, False),
    ((2, 6, 11, 13, 10, 3, 3, 1, 1, 2, 1), (1, 1), 2, False, True),
    ((1, 8, 30, 33, 64, 4, 3, 1, 1, 1, 2), (1, 1), 1, False, False),
    ((2, 3, 64, 96, 64, 6, 7, 0, 3, 1, 1), (1, 1), 1, False, False),   # 5-row, 6-column halo
]


@pytest.mark.parametrize("case", C2I_CASES, ids=[f"c2i{i}" for i in range(len(C2I_CASES))])
def test_few_channel_bwd_data_parity(cg, case):
    (N, C, H, Wd, K, R, S, ph, pw, sh, sw), dil, groups, flip, epi = case
    dh, dw_ = dil
    P = (H + 2 * ph - dh * (R - 1) - 1) // sh + 1
    Q = (Wd + 2 * pw - dw_ * (S - 1) - 1) // sw + 1
    g = torch.Generator().manual_seed(9700 + C2I_CASES.index(case))
    dy = torch.randn(N, K, P, Q, generator=g)
    w = torch.randn(K, C // groups, R, S, generator=g)
    bc = torch.randn(C, generator=g) if epi else None
    dx0 = torch.randn(N, C, H, Wd, generator=g)
    pad, st = (ph, pw), (sh, sw)
    dx = dx0.to(DEV) if epi else _poisoned((N, C, H, Wd), torch.float32)
    cg.conv2d_bwd_data(dy.to(DEV), w.to(DEV), (H, Wd), pad, st, out=dx, bias=bc.to(DEV) if epi else None,
                       beta=0.5 if epi else 0.0, flip=flip, dilation=dil, groups=groups)
    cg.conv2d_device_status()
    ref = oracle.conv2d_bwd_data_ex(dy, w, (H, Wd), bc, 0.5 if epi else 0.0, dx0 if epi else None, pad, st,
                                    flip, dil, groups)
    pb = W.Conv2dProblem(N, C, H, Wd, K, R, S, ph, pw, sh, sw, "f32")
    scale = float(dy.abs().max()) * float(w.abs().max())
    _check_plain(pb, dx.double().cpu().numpy(), ref, scale, (K // groups) * R * S, f"{case}")
    # deterministic: a second call gives the same bits
    dx2 = dx0.to(DEV) if epi else _poisoned((N, C, H, Wd), torch.float32)
    cg.conv2d_bwd_data(dy.to(DEV), w.to(DEV), (H, Wd), pad, st, out=dx2, bias=bc.to(DEV) if epi else None,
                       beta=0.5 if epi else 0.0, flip=flip, dilation=dil, groups=groups)
    assert torch.equal(dx, dx2)


# Backward-filter with few input channels (fp32): the TMEM-built filter-gradient path on
# stem-like shapes.  Cases: strides, dilation, K up to 128, groups, convolution mode, add-to
# (beta) and both bias gradients, ragged rows; fixed-order split sums (bitwise repeatable).
FC_CASES = [
    # (N, C, H, W, K, R, S, ph, pw, sh, sw), (dh, dw), groups, flip, epilogue
    ((2, 3, 32, 40, 16, 7, 7, 3, 3, 2, 2), (1, 1), 1, False, False),   # the stem's shape, small
    ((1, 4, 20, 24, 40, 3, 3, 1, 1, 1, 1), (1, 1), 1, True, True),
    ((1, 2, 16, 36, 9, 3, 3, 2, 2, 1, 1), (2, 2), 1, False, True),
    ((1, 2, 12, 16, 128, 3, 3, 1, 1, 1, 1), (1, 1), 1, False, False),
    ((2, 8, 12, 16, 12, 3, 3, 1, 1, 1, 1), (1, 1), 2, True, False),
    ((1, 16, 14, 18, 24, 3, 3, 1, 1, 1, 1), (1, 1), 4, True, True),   # four groups, add-to: diagonal blocks only
    ((1, 1, 9, 140, 5, 1, 5, 0, 2, 1, 1), (1, 1), 1, False, True),
    ((3, 3, 64, 64, 64, 7, 7, 3, 3, 2, 2), (1, 1), 1, False, False),
]


@pytest.mark.parametrize("case", FC_CASES, ids=[f"fc{i}" for i in range(len(FC_CASES))])
def test_few_channel_bwd_filter_parity(cg, case):
    (N, C, H, Wd, K, R, S, ph, pw, sh, sw), dil, groups, flip, epi = case
    dh, dw_ = dil
    P = (H + 2 * ph - dh * (R - 1) - 1) // sh + 1
    Q = (Wd + 2 * pw - dw_ * (S - 1) - 1) // sw + 1
    g = torch.Generator().manual_seed(9800 + FC_CASES.index(case))
    x = torch.randn(N, C, H, Wd, generator=g)
    dy = torch.randn(N, K, P, Q, generator=g)
    dw0 = torch.randn(K, C // groups, R, S, generator=g)
    pad, st = (ph, pw), (sh, sw)
    beta = 0.5 if epi else 0.0
    dw = dw0.to(DEV) if epi else _poisoned((K, C // groups, R, S), torch.float32)
    dbk = torch.zeros(K, device=DEV) if epi else None
    dbc = torch.zeros(C, device=DEV) if epi else None
    cg.conv2d_bwd_filter(x.to(DEV), dy.to(DEV), (R, S), pad, st, out=dw, beta=beta, flip=flip, dilation=dil,
                         groups=groups, db_k=dbk, db_c=dbc)
    cg.conv2d_device_status()
    ref = oracle.conv2d_bwd_filter_ex(x, dy, (R, S), beta, dw0 if epi else None, pad, st, flip, dil, groups)
    pb = W.Conv2dProblem(N, C, H, Wd, K, R, S, ph, pw, sh, sw, "f32")
    scale = float(x.abs().max()) * float(dy.abs().max())
    _check_plain(pb, dw.double().cpu().numpy(), ref, scale, N * P * Q, f"{case}")
    if epi:
        _check_plain(pb, dbk.double().cpu().numpy(), oracle.channel_sum(dy), float(dy.abs().max()), N * P * Q,
                     f"{case}/db_k")
        _check_plain(pb, dbc.double().cpu().numpy(), oracle.channel_sum(x), float(x.abs().max()), N * H * Wd,
                     f"{case}/db_c")
    dw2 = dw0.to(DEV) if epi else _poisoned((K, C // groups, R, S), torch.float32)
    cg.conv2d_bwd_filter(x.to(DEV), dy.to(DEV), (R, S), pad, st, out=dw2, beta=beta, flip=flip, dilation=dil,
                         groups=groups)
    assert torch.equal(dw, dw2)  # deterministic (fixed-order split sums)

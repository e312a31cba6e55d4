"""Pins for the fp64 CPU oracle's 3-D (NCDHW) ops (CPU only).

Semantics (page title): Apache MXNet mkldnn_deconvolution.cc -- SupportMKLDNNDeconv: kernels
of one to three spatial dims on an input of two more dims; DeconvDescCreator: one stride, pad
and dilation per spatial dim.

The 3-D oracle is trusted only after it agrees with things other than itself:
hand-counted all-ones values (tests/golden/box_ones_3d.txt); depth-1 problems equal the
pinned 2-D oracle; depth-only problems equal a 1-D cross-correlation run through the
2-D oracle; every problem equals the sum over depth taps of 2-D convolutions of depth
slices (a decomposition of the definition, evaluated with the pinned 2-D oracle); the
adjoint identity across the three ops; and PyTorch CPU fp64 (conv3d and its autograd
gradients) as a library witness.  The last group compiles copies of the C oracle with a
planted mistake each and checks that the pins reject every one.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")
ORACLE_DIR = os.path.dirname(os.path.abspath(oracle.__file__))
RNG = np.random.default_rng(20261203)

# N C D H W K T R S pad stride dilation groups: no two extents equal where that can hide an
# index swap; ragged output sizes; every pad / stride / dilation > 1 somewhere.
CASES = [
    (2, 3, 5, 6, 7, 4, 3, 2, 3, (1, 0, 1), (1, 1, 1), (1, 1, 1), 1),
    (1, 4, 9, 5, 6, 6, 2, 3, 2, (2, 1, 0), (2, 1, 2), (2, 1, 1), 2),
    (2, 2, 7, 8, 5, 3, 3, 2, 2, (1, 2, 1), (3, 2, 1), (1, 2, 2), 1),
    (1, 6, 6, 4, 9, 4, 2, 2, 3, (0, 1, 2), (1, 2, 1), (3, 1, 2), 2),
]


def _out3(case):
    N, C, D, H, W, K, T, R, S, pad, stride, dil, g = case
    return tuple(oracle.output_dim_dilated(i, p, k, s, d)
                 for i, p, k, s, d in zip((D, H, W), pad, (T, R, S), stride, dil))


def _tensors(case, rng):
    N, C, D, H, W, K, T, R, S, pad, stride, dil, g = case
    Z, P, Q = _out3(case)
    assert min(Z, P, Q) >= 1
    x = rng.standard_normal((N, C, D, H, W))
    w = rng.standard_normal((K, C // g, T, R, S))
    dy = rng.standard_normal((N, K, Z, P, Q))
    return x, w, dy


def _fwd(x, w, case):
    return oracle.conv3d_fwd(x, w, case[9], case[10], case[11], case[12])


def _bwd_data(dy, w, case):
    return oracle.conv3d_bwd_data(dy, w, case[2:5], case[9], case[10], case[11], case[12])


def _bwd_filter(x, dy, case):
    return oracle.conv3d_bwd_filter(x, dy, case[6:9], case[9], case[10], case[11], case[12])


def _close(a, b, rtol=1e-12):
    a, b = np.asarray(a), np.asarray(b)
    return a.shape == b.shape and bool(np.all(np.abs(a - b) <= rtol * (1.0 + np.abs(b).max())))


def _load_golden(name):
    tens = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(":", 1)
            shape, data = rest.split("|")
            shape = tuple(int(v) for v in shape.split(","))
            tens[key.strip()] = np.array([float(v) for v in data.split()]).reshape(shape)
    return tens


# --------------------------------------------------------------------------- pin checks
# Each returns True when the pin holds; the tests assert them on the real oracle, and the
# planted-mistake tests assert that at least one fails on each mutated copy.

def _golden_ok():
    t = _load_golden("box_ones_3d.txt")
    ok = np.array_equal(oracle.conv3d_fwd(np.ones((1, 1, 3, 3, 4)), np.ones((1, 1, 3, 3, 3)), 1, 1, 1), t["yA"])
    caseB = dict(pad=(1, 0, 0), stride=(2, 1, 1), dilation=(2, 1, 1))
    ok &= np.array_equal(oracle.conv3d_fwd(np.ones((1, 1, 5, 1, 1)), np.ones((1, 1, 2, 1, 1)), **caseB), t["yB"])
    ok &= np.array_equal(oracle.conv3d_bwd_data(np.ones((1, 1, 3, 1, 1)), np.ones((1, 1, 2, 1, 1)), (5, 1, 1),
                                                **caseB), t["dxB"])
    ok &= np.array_equal(oracle.conv3d_bwd_filter(np.ones((1, 1, 5, 1, 1)), np.ones((1, 1, 3, 1, 1)), (2, 1, 1),
                                                  **caseB), t["dwB"])
    return bool(ok)


def _depth_one_ok(case, rng):
    """D = T = 1, no depth pad: the 3-D ops are the 2-D ops on the single depth slice."""
    N, C, _, H, W, K, _, R, S, pad, stride, dil, g = case
    c1 = (N, C, 1, H, W, K, 1, R, S, (0,) + pad[1:], (1,) + stride[1:], (1,) + dil[1:], g)
    x, w, dy = _tensors(c1, rng)
    p2, s2, d2 = pad[1:], stride[1:], dil[1:]
    ok = _close(_fwd(x, w, c1)[:, :, 0], oracle.conv2d_fwd_ex(x[:, :, 0], w[:, :, 0], pad=p2, stride=s2,
                                                             dilation=d2, groups=g))
    ok &= _close(_bwd_data(dy, w, c1)[:, :, 0],
                 oracle.conv2d_bwd_data_ex(dy[:, :, 0], w[:, :, 0], (H, W), pad=p2, stride=s2, dilation=d2,
                                           groups=g))
    ok &= _close(_bwd_filter(x, dy, c1)[:, :, 0],
                 oracle.conv2d_bwd_filter_ex(x[:, :, 0], dy[:, :, 0], (R, S), pad=p2, stride=s2, dilation=d2,
                                             groups=g))
    return bool(ok)


def _depth_only_ok(case, rng):
    """H = W = R = S = 1: a 1-D cross-correlation along depth, run through the 2-D oracle as
    (D, 1) images with a (T, 1) filter."""
    N, C, D, _, _, K, T, _, _, pad, stride, dil, g = case
    c1 = (N, C, D, 1, 1, K, T, 1, 1, (pad[0], 0, 0), (stride[0], 1, 1), (dil[0], 1, 1), g)
    x, w, dy = _tensors(c1, rng)
    kw = dict(pad=(pad[0], 0), stride=(stride[0], 1), dilation=(dil[0], 1), groups=g)
    ok = _close(_fwd(x, w, c1)[..., 0], oracle.conv2d_fwd_ex(x[..., 0], w[..., 0], **kw))
    ok &= _close(_bwd_data(dy, w, c1)[..., 0], oracle.conv2d_bwd_data_ex(dy[..., 0], w[..., 0], (D, 1), **kw))
    ok &= _close(_bwd_filter(x, dy, c1)[..., 0], oracle.conv2d_bwd_filter_ex(x[..., 0], dy[..., 0], (T, 1), **kw))
    return bool(ok)


def _depth_slices_ok(case, rng):
    """y[:, :, z] = sum over depth taps t of conv2d(x[:, :, z*sd - pd + t*dd], w[:, :, t]), slices
    outside the input being zero; the two gradients decompose the same way."""
    N, C, D, H, W, K, T, R, S, pad, stride, dil, g = case
    Z, P, Q = _out3(case)
    x, w, dy = _tensors(case, rng)
    kw = dict(pad=pad[1:], stride=stride[1:], dilation=dil[1:], groups=g)
    y = np.zeros((N, K, Z, P, Q))
    dx = np.zeros((N, C, D, H, W))
    dw = np.zeros(w.shape)
    for z in range(Z):
        for t in range(T):
            zi = z * stride[0] - pad[0] + t * dil[0]
            if not 0 <= zi < D:
                continue
            y[:, :, z] += oracle.conv2d_fwd_ex(x[:, :, zi], w[:, :, t], **kw)
            dx[:, :, zi] += oracle.conv2d_bwd_data_ex(dy[:, :, z], w[:, :, t], (H, W), **kw)
            dw[:, :, t] += oracle.conv2d_bwd_filter_ex(x[:, :, zi], dy[:, :, z], (R, S), **kw)
    return _close(_fwd(x, w, case), y) and _close(_bwd_data(dy, w, case), dx) and \
        _close(_bwd_filter(x, dy, case), dw)


def _adjoint_ok(case, rng):
    """<fwd(x, w), dy> = <x, bwd_data(dy, w)> = <w, bwd_filter(x, dy)>."""
    x, w, dy = _tensors(case, rng)
    a = np.vdot(_fwd(x, w, case), dy)
    b = np.vdot(x, _bwd_data(dy, w, case))
    c = np.vdot(w, _bwd_filter(x, dy, case))
    return abs(a - b) <= 1e-11 * abs(a) and abs(a - c) <= 1e-11 * abs(a)


def _pins_pass():
    ok = _golden_ok()
    for i, case in enumerate(CASES):
        rng = np.random.default_rng(100 + i)
        ok &= _depth_one_ok(case, rng) and _depth_only_ok(case, rng) and _depth_slices_ok(case, rng) \
            and _adjoint_ok(case, rng)
    return bool(ok)


# --------------------------------------------------------------------------- the pins
def test_output_dims_of_the_cases():
    """The cases are ragged and every output extent is positive (window enumeration)."""
    for case in CASES:
        N, C, D, H, W, K, T, R, S, pad, stride, dil, g = case
        for i, p, k, s, d, o in zip((D, H, W), pad, (T, R, S), stride, dil, _out3(case)):
            ext = d * (k - 1) + 1
            assert o == sum(1 for start in range(-p, i + p) if (start + p) % s == 0 and start + ext - 1 <= i - 1 + p)


def test_golden_box_ones_3d():
    assert _golden_ok()


@pytest.mark.parametrize("case", CASES)
def test_depth_one_equals_2d(case):
    assert _depth_one_ok(case, RNG)


@pytest.mark.parametrize("case", CASES)
def test_depth_only_equals_1d(case):
    assert _depth_only_ok(case, RNG)


@pytest.mark.parametrize("case", CASES)
def test_sum_over_depth_taps_of_2d_slices(case):
    assert _depth_slices_ok(case, RNG)


@pytest.mark.parametrize("case", CASES)
def test_adjoint_identity_3d(case):
    assert _adjoint_ok(case, RNG)


@pytest.mark.parametrize("case", CASES)
def test_torch_cpu_fp64_witness_3d(case):
    torch = pytest.importorskip("torch")
    N, C, D, H, W, K, T, R, S, pad, stride, dil, g = case
    x, w, dy = _tensors(case, RNG)
    xt = torch.tensor(x, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    yt = torch.nn.functional.conv3d(xt, wt, stride=stride, padding=pad, dilation=dil, groups=g)
    yt.backward(torch.tensor(dy))
    assert _close(_fwd(x, w, case), yt.detach().numpy(), 1e-11)
    assert _close(_bwd_data(dy, w, case), xt.grad.numpy(), 1e-11)
    assert _close(_bwd_filter(x, dy, case), wt.grad.numpy(), 1e-11)


@pytest.mark.parametrize("case", [c for c in CASES if c[12] == 1])
def test_sampled_equals_full_3d(case):
    """The sampled evaluators (full-size parity) agree bit for bit with the full ops."""
    x, w, dy = _tensors(case, RNG)
    dims = oracle.conv3d_dims(x.shape, w.shape, case[9], case[10], case[11])
    y, dx, dw = _fwd(x, w, case), _bwd_data(dy, w, case), _bwd_filter(x, dy, case)
    for full, fn, a, b in ((y, oracle.conv3d_fwd_at, x, w), (dx, oracle.conv3d_bwd_data_at, dy, w),
                           (dw, oracle.conv3d_bwd_filter_at, x, dy)):
        idx = RNG.choice(full.size, size=min(40, full.size), replace=False)
        assert np.array_equal(fn(a, b, dims, idx), full.reshape(-1)[idx])


# --------------------------------------------------------------------------- planted mistakes
# Each entry: (function in conv3d_oracle.c, text there, replacement).  Every replacement keeps
# all reads in bounds (reads go through the zero-padding helper or the reader test).
MUTATIONS = {
    "fwd_depth_dilation_dropped": ("static double fwd3_one", "t * g->dd", "t"),
    "fwd_depth_pad_sign": ("static double fwd3_one", "- g->pd +", "+ g->pd +"),
    "fwd_filter_taps_swapped": ("static double fwd3_one", "w[IDX5(k, c, t, r, s,", "w[IDX5(k, c, r % g->T, t % g->R, s,"),
    "bwd_data_depth_stride_ignored": ("static double bwd_data3_one", "reader(z, t, g->pd, g->sd,", "reader(z, t, g->pd, 1,"),
    "bwd_data_row_dilation_dropped": ("static double bwd_data3_one", "reader(h, r, g->ph, g->sh, g->dh,",
                                      "reader(h, r, g->ph, g->sh, 1,"),
    "reader_divisibility_dropped": ("static inline int reader", "if (t < 0 || t % stride != 0)", "if (t < 0)"),
    "bwd_filter_column_dilation_dropped": ("static double bwd_filter3_one", "q * g->sw - g->pw + s * g->dw",
                                           "q * g->sw - g->pw + s"),
    "pads_swapped": ("static geom3 make_geom", "q.pd = g[9]; q.ph = g[10];", "q.pd = g[10]; q.ph = g[9];"),
}


def _mutant_lib(tmp_path, name, mutation):
    with open(os.path.join(ORACLE_DIR, "conv3d_oracle.c")) as f:
        src = f.read()
    if mutation is not None:
        marker, old, new = mutation
        at = src.index(marker)
        pos = src.index(old, at)
        src = src[:pos] + new + src[pos + len(old):]
    c3 = tmp_path / f"{name}.c"
    c3.write_text(src)
    so = tmp_path / f"lib{name}.so"
    subprocess.check_call(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c99", "-o", str(so),
                           os.path.join(ORACLE_DIR, "conv2d_oracle.c"), str(c3)])
    return oracle._bind(ctypes.CDLL(str(so)))


def test_pins_accept_unmutated_copy(tmp_path, monkeypatch):
    monkeypatch.setattr(oracle, "_lib", _mutant_lib(tmp_path, "unmutated", None))
    assert _pins_pass()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_planted_mistake(tmp_path, monkeypatch, name):
    monkeypatch.setattr(oracle, "_lib", _mutant_lib(tmp_path, name, MUTATIONS[name]))
    assert not _pins_pass()

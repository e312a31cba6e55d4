"""Pins for the fp64 CPU oracle (CPU only).

The oracle is trusted only after it agrees with things other than itself:
hand-derived golden values, closed forms (1x1 conv = matmul, delta filter =
shifted copy), the adjoint identity linking the three ops, the transpose of
the dense linear operator built by brute force, a scatter-form deconvolution,
window enumeration for P/Q, and an independent library witness (PyTorch CPU
fp64).  The last group plants mistakes in small pure-Python convolutions and
checks that the pins catch each one.

Semantics pinned (page titles): Apache SystemDS LibMatrixCuDNNConvolutionAlgorithm.java
-- NCHW / KCRS, cross-correlation, dilation 1, the 13 descriptor integers;
Apache MXNet mkldnn_deconvolution.cc -- deconvolution forward = convolution
backward-data with the weight read as (deconv_in, deconv_out, h, w).
"""
import itertools
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(20261202)


def _load_golden(name):
    vals, tens = {}, {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(":", 1)
            if "|" in rest:
                shape, data = rest.split("|")
                shape = tuple(int(v) for v in shape.split(","))
                tens[key.strip()] = np.array([float(v) for v in data.split()]).reshape(shape)
            else:
                vals[key.strip()] = int(rest)
    return vals, tens


# --------------------------------------------------------------------------- P/Q
def _count_windows(inp, pad, k, stride):
    """Number of window start positions p >= 0 whose k taps p*stride-pad .. p*stride-pad+k-1
    all lie inside the zero-padded input [-pad, inp+pad)."""
    n = 0
    p = 0
    while p * stride - pad + k - 1 <= inp - 1 + pad:
        n += 1
        p += 1
    return n


def test_output_dim_matches_window_enumeration():
    for inp, pad, k, st in itertools.product(range(1, 65), range(0, 4), range(1, 8), range(1, 4)):
        assert oracle.output_dim(inp, pad, k, st) == _count_windows(inp, pad, k, st), (inp, pad, k, st)


def test_output_dim_config_values():
    # P=Q for the six workloads: 8, 56, 28, 14, 112, 16 (deconv: H=32 -> P=16).
    assert oracle.output_dim(8, 1, 3, 1) == 8
    assert oracle.output_dim(56, 1, 3, 1) == 56
    assert oracle.output_dim(56, 1, 3, 2) == 28
    assert oracle.output_dim(14, 0, 1, 1) == 14
    assert oracle.output_dim(224, 3, 7, 2) == 112
    assert oracle.output_dim(32, 1, 4, 2) == 16
    assert oracle.output_dim(33, 1, 4, 2) == 16   # H is not unique for stride > 1
    assert oracle.output_dim(2, 0, 3, 1) == 0     # filter larger than padded input
    assert oracle.output_dim(0, 0, 1, 1) == -1


# --------------------------------------------------------------------------- golden
def test_golden_box_filter_counts():
    v, t = _load_golden("box_ones_4x5.txt")
    x = np.ones((1, 1, v["H"], v["W"]))
    w = np.ones((1, 1, v["R"], v["S"]))
    pad = v["pad"]
    assert np.array_equal(oracle.conv2d_fwd(x, w, pad, 1), t["y_stride1"])
    assert np.array_equal(oracle.conv2d_fwd(x, w, pad, 2), t["y_stride2"])
    dy2 = np.ones((1, 1, 2, 3))
    assert np.array_equal(oracle.conv2d_bwd_data(dy2, w, (v["H"], v["W"]), pad, 2), t["dx_stride2"])
    dy1 = np.ones((1, 1, 4, 5))
    assert np.array_equal(oracle.conv2d_bwd_filter(x, dy1, (3, 3), pad, 1), t["dw_stride1"])


def test_golden_nonsymmetric():
    _, t = _load_golden("nonsymmetric.txt")
    assert np.array_equal(oracle.conv2d_fwd(t["x1"], t["wa"]), t["ya"])
    assert np.array_equal(oracle.conv2d_fwd(t["x1"], t["wb"]), t["yb"])
    assert np.array_equal(oracle.conv2d_fwd(t["x2"], t["wc"]), t["yc"])


# --------------------------------------------------------------------------- closed forms
@pytest.mark.parametrize("N,C,H,W,K,stride", [(3, 5, 4, 6, 7, 1), (2, 8, 7, 5, 3, 2), (2, 256, 14, 14, 16, 1)])
def test_1x1_is_matmul(N, C, H, W, K, stride):
    x = RNG.standard_normal((N, C, H, W))
    w = RNG.standard_normal((K, C, 1, 1))
    y = oracle.conv2d_fwd(x, w, 0, stride)
    ref = np.einsum("kc,nchw->nkhw", w[:, :, 0, 0], x[:, :, ::stride, ::stride])
    assert y.shape == ref.shape
    assert np.max(np.abs(y - ref)) <= 1e-13 * max(1.0, np.max(np.abs(ref)))


@pytest.mark.parametrize("H,W,R,S,ph,pw,sh,sw", [
    (7, 9, 3, 3, 1, 1, 1, 1), (8, 6, 3, 5, 1, 2, 2, 1), (9, 9, 7, 7, 3, 3, 2, 2), (5, 11, 2, 4, 0, 1, 3, 2)])
def test_delta_filter_is_shifted_padded_copy(H, W, R, S, ph, pw, sh, sw):
    N, C = 2, 3
    x = RNG.standard_normal((N, C, H, W))
    xp = np.pad(x, ((0, 0), (0, 0), (ph, ph), (pw, pw)))
    P = oracle.output_dim(H, ph, R, sh)
    Q = oracle.output_dim(W, pw, S, sw)
    for r0, s0 in [(0, 0), (R - 1, S - 1), (R // 2, S - 1)]:
        w = np.zeros((C, C, R, S))
        for c in range(C):
            w[c, c, r0, s0] = 1.0
        y = oracle.conv2d_fwd(x, w, (ph, pw), (sh, sw))
        ref = xp[:, :, r0:r0 + sh * (P - 1) + 1:sh, s0:s0 + sw * (Q - 1) + 1:sw]
        assert np.array_equal(y, ref)  # bitwise: one product by 1.0 per output


ADJ_CASES = [
    # N, C, H, W, K, R, S, ph, pw, sh, sw
    (2, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1),
    (1, 2, 7, 9, 3, 3, 2, 0, 1, 2, 1),
    (2, 3, 9, 8, 2, 5, 3, 2, 1, 3, 2),   # trailing rows not covered by any window
    (1, 4, 6, 6, 3, 4, 4, 1, 1, 2, 2),   # deconvolution-style 4x4 / 2
    (2, 1, 5, 13, 2, 5, 13, 0, 0, 1, 1),  # H == R and W == S (conv1d-like)
]


@pytest.mark.parametrize("case", ADJ_CASES)
def test_adjoint_identity(case):
    N, C, H, W, K, R, S, ph, pw, sh, sw = case
    P, Q = oracle.output_dim(H, ph, R, sh), oracle.output_dim(W, pw, S, sw)
    x = RNG.standard_normal((N, C, H, W))
    w = RNG.standard_normal((K, C, R, S))
    dy = RNG.standard_normal((N, K, P, Q))
    a = np.vdot(oracle.conv2d_fwd(x, w, (ph, pw), (sh, sw)), dy)
    b = np.vdot(x, oracle.conv2d_bwd_data(dy, w, (H, W), (ph, pw), (sh, sw)))
    c = np.vdot(w, oracle.conv2d_bwd_filter(x, dy, (R, S), (ph, pw), (sh, sw)))
    assert abs(a - b) <= 1e-12 * abs(a) and abs(a - c) <= 1e-12 * abs(a)


@pytest.mark.parametrize("case", [(1, 2, 5, 4, 3, 3, 2, 1, 0, 2, 1), (2, 1, 6, 7, 2, 3, 3, 1, 1, 1, 2)])
def test_dense_operator_transpose(case):
    """Build the matrices of x -> y and w -> y column by column from unit vectors
    and check that bwd_data / bwd_filter apply their transposes."""
    N, C, H, W, K, R, S, ph, pw, sh, sw = case
    P, Q = oracle.output_dim(H, ph, R, sh), oracle.output_dim(W, pw, S, sw)
    w = RNG.standard_normal((K, C, R, S))
    x = RNG.standard_normal((N, C, H, W))
    dy = RNG.standard_normal((N, K, P, Q))
    A = np.zeros((N * K * P * Q, N * C * H * W))
    for j in range(A.shape[1]):
        e = np.zeros(N * C * H * W)
        e[j] = 1.0
        A[:, j] = oracle.conv2d_fwd(e.reshape(N, C, H, W), w, (ph, pw), (sh, sw)).ravel()
    B = np.zeros((N * K * P * Q, K * C * R * S))
    for j in range(B.shape[1]):
        e = np.zeros(K * C * R * S)
        e[j] = 1.0
        B[:, j] = oracle.conv2d_fwd(x, e.reshape(K, C, R, S), (ph, pw), (sh, sw)).ravel()
    dx = oracle.conv2d_bwd_data(dy, w, (H, W), (ph, pw), (sh, sw)).ravel()
    dw = oracle.conv2d_bwd_filter(x, dy, (R, S), (ph, pw), (sh, sw)).ravel()
    assert np.max(np.abs(dx - A.T @ dy.ravel())) <= 1e-13 * max(1.0, np.max(np.abs(dx)))
    assert np.max(np.abs(dw - B.T @ dy.ravel())) <= 1e-13 * max(1.0, np.max(np.abs(dw)))


@pytest.mark.parametrize("N,Ci,Co,Hi,R,pad,stride,Ho", [
    (2, 5, 3, 4, 4, 1, 2, 8),    # the deconvolution workload's geometry, scaled down
    (1, 3, 2, 5, 4, 1, 2, 11),   # Ho = 10 and 11 both give Hi = 5 under the floor
    (2, 2, 4, 6, 3, 1, 1, 6),
    (1, 4, 2, 3, 7, 3, 2, 6),
])
def test_deconv_scatter_equals_bwd_data(N, Ci, Co, Hi, R, pad, stride, Ho):
    if oracle.output_dim(Ho, pad, R, stride) != Hi:
        pytest.skip("inconsistent geometry")
    inp = RNG.standard_normal((N, Ci, Hi, Hi))
    wt = RNG.standard_normal((Ci, Co, R, R))     # (deconv_in, deconv_out, h, w)
    sc = oracle.deconv2d_fwd_scatter(inp, wt, (Ho, Ho), pad, stride)
    ga = oracle.conv2d_bwd_data(inp, wt, (Ho, Ho), pad, stride)  # conv view: K = Ci, C = Co
    assert np.max(np.abs(sc - ga)) <= 1e-13 * max(1.0, np.max(np.abs(sc)))


def test_uncovered_rows_are_zero():
    # H=W=10, pad 0, R=3, stride 2 -> P=Q=4: windows start at rows 0,2,4,6 and read rows
    # 0..8; row 9 (and column 9) is never read, so its gradient must be exactly 0.
    x_hw = (10, 10)
    P = oracle.output_dim(10, 0, 3, 2)
    assert P == 4
    dy = RNG.standard_normal((1, 2, P, P))
    w = RNG.standard_normal((2, 3, 3, 3))
    dx = oracle.conv2d_bwd_data(dy, w, x_hw, 0, 2)
    assert np.all(dx[:, :, 9, :] == 0.0) and np.all(dx[:, :, :, 9] == 0.0)
    assert np.any(dx[:, :, 8, :] != 0.0)


def test_sampled_equals_full():
    N, C, H, W, K, R, S, ph, pw, sh, sw = (2, 3, 9, 7, 4, 3, 2, 1, 1, 2, 1)
    P, Q = oracle.output_dim(H, ph, R, sh), oracle.output_dim(W, pw, S, sw)
    dims = (N, C, H, W, K, R, S, ph, pw, sh, sw, P, Q)
    x = RNG.standard_normal((N, C, H, W))
    w = RNG.standard_normal((K, C, R, S))
    dy = RNG.standard_normal((N, K, P, Q))
    y = oracle.conv2d_fwd(x, w, (ph, pw), (sh, sw))
    dx = oracle.conv2d_bwd_data(dy, w, (H, W), (ph, pw), (sh, sw))
    dw = oracle.conv2d_bwd_filter(x, dy, (R, S), (ph, pw), (sh, sw))
    for full, fn, a, b in [(y, oracle.conv2d_fwd_at, x, w), (dx, oracle.conv2d_bwd_data_at, dy, w),
                           (dw, oracle.conv2d_bwd_filter_at, x, dy)]:
        idx = RNG.choice(full.size, size=min(25, full.size), replace=False)
        assert np.array_equal(fn(a, b, dims, idx), full.ravel()[idx])


# --------------------------------------------------------------------------- library witness
@pytest.mark.parametrize("case", ADJ_CASES[:4])
def test_torch_cpu_fp64_witness(case):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    N, C, H, W, K, R, S, ph, pw, sh, sw = case
    P, Q = oracle.output_dim(H, ph, R, sh), oracle.output_dim(W, pw, S, sw)
    x = RNG.standard_normal((N, C, H, W))
    w = RNG.standard_normal((K, C, R, S))
    dy = RNG.standard_normal((N, K, P, Q))
    tx, tw, tdy = (torch.from_numpy(a) for a in (x, w, dy))
    y_ref = F.conv2d(tx, tw, stride=(sh, sw), padding=(ph, pw)).numpy()
    dx_ref = torch.nn.grad.conv2d_input((N, C, H, W), tw, tdy, stride=(sh, sw), padding=(ph, pw)).numpy()
    dw_ref = torch.nn.grad.conv2d_weight(tx, (K, C, R, S), tdy, stride=(sh, sw), padding=(ph, pw)).numpy()
    for got, ref in [(oracle.conv2d_fwd(x, w, (ph, pw), (sh, sw)), y_ref),
                     (oracle.conv2d_bwd_data(dy, w, (H, W), (ph, pw), (sh, sw)), dx_ref),
                     (oracle.conv2d_bwd_filter(x, dy, (R, S), (ph, pw), (sh, sw)), dw_ref)]:
        assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


# --------------------------------------------------------------------------- planted mistakes
def _py_fwd(x, w, pad, stride, mistake=None):
    """Tiny pure-Python forward with an optional planted mistake."""
    N, C, H, W = x.shape
    K, _, R, S = w.shape
    ph, pw = pad
    sh, sw = stride
    P = (H + 2 * ph - R) // sh + 1
    Q = (W + 2 * pw - S) // sw + 1
    y = np.zeros((N, K, P, Q))
    for n, k, p, q, c, r, s in itertools.product(range(N), range(K), range(P), range(Q),
                                                 range(C), range(R), range(S)):
        rr, ss = (R - 1 - r, S - 1 - s) if mistake == "flip" else (r, s)
        h = p * sh - ph + rr
        ww = q * sw - (0 if mistake == "left_pad_dropped" else pw) + ss
        if mistake == "transposed_filter":
            wv = w.reshape(C, K, R, S)[c, k, r, s]
        else:
            wv = w[k, c, r, s]
        if 0 <= h < H and 0 <= ww < W:
            y[n, k, p, q] += x[n, c, h, ww] * wv
    return y


def _py_bwd_data(dy, w, x_hw, pad, stride, mistake=None):
    N, K, P, Q = dy.shape
    _, C, R, S = w.shape
    H, W = x_hw
    ph, pw = pad
    sh, sw = stride
    dx = np.zeros((N, C, H, W))
    for n, k, p, q, c, r, s in itertools.product(range(N), range(K), range(P), range(Q),
                                                 range(C), range(R), range(S)):
        h = p * sh - ph + r
        ww = q * sw - pw + s
        if mistake == "swap_rs":
            wv = w[k, c, s % R, r % S]
        else:
            wv = w[k, c, r, s]
        if mistake == "stride_ignored":
            h, ww = p - ph + r, q - pw + s
        if 0 <= h < H and 0 <= ww < W:
            dx[n, c, h, ww] += dy[n, k, p, q] * wv
    return dx


def _pins_pass(fwd, bwd_data):
    """Run the cheap pins against a (fwd, bwd_data) pair; True if all hold."""
    _, t = _load_golden("nonsymmetric.txt")
    ok = True
    ok &= np.array_equal(fwd(t["x1"], t["wa"], (0, 0), (1, 1)), t["ya"])
    ok &= np.array_equal(fwd(t["x1"], t["wb"], (0, 0), (1, 1)), t["yb"])
    ok &= np.array_equal(fwd(t["x2"], t["wc"], (0, 0), (1, 1)), t["yc"])
    v, g = _load_golden("box_ones_4x5.txt")
    ones = np.ones((1, 1, 4, 5))
    ok &= np.array_equal(fwd(ones, np.ones((1, 1, 3, 3)), (1, 1), (2, 2)), g["y_stride2"])
    rng = np.random.default_rng(7)
    for case in ADJ_CASES[1:3]:
        N, C, H, W, K, R, S, ph, pw, sh, sw = case
        P, Q = (H + 2 * ph - R) // sh + 1, (W + 2 * pw - S) // sw + 1
        x = rng.standard_normal((N, C, H, W))
        w = rng.standard_normal((K, C, R, S))
        dy = rng.standard_normal((N, K, P, Q))
        a = np.vdot(fwd(x, w, (ph, pw), (sh, sw)), dy)
        b = np.vdot(x, bwd_data(dy, w, (H, W), (ph, pw), (sh, sw)))
        ok &= abs(a - b) <= 1e-12 * abs(a)
    return bool(ok)


def test_pins_accept_correct_python_reference():
    assert _pins_pass(_py_fwd, _py_bwd_data)


@pytest.mark.parametrize("mistake", ["flip", "left_pad_dropped", "transposed_filter"])
def test_pins_catch_planted_fwd_mistake(mistake):
    assert not _pins_pass(lambda *a: _py_fwd(*a, mistake=mistake), _py_bwd_data)


@pytest.mark.parametrize("mistake", ["swap_rs", "stride_ignored"])
def test_pins_catch_planted_bwd_data_mistake(mistake):
    assert not _pins_pass(_py_fwd, lambda *a: _py_bwd_data(*a, mistake=mistake))


# --------------------------------------------------------------------------- fused epilogues
# Page "mkldnn_deconvolution.cc": optional bias on the deconvolution output, output request
# write / add-to, bias gradient in the backward-weights pass.  Pinned by closed forms (zero
# operands), by the derivative identity linking a bias to its gradient, and by PyTorch CPU
# fp64 (conv2d / conv_transpose2d with bias).
EPI = (2, 3, 5, 7, 4, 3, 2, 1, 0, 2, 1)  # N C H W K R S ph pw sh sw: no two sizes equal


def _epi_shapes():
    N, C, H, W, K, R, S, ph, pw, sh, sw = EPI
    return N, C, H, W, K, R, S, ph, pw, sh, sw, oracle.output_dim(H, ph, R, sh), oracle.output_dim(W, pw, S, sw)


def test_epilogue_closed_forms_with_zero_operands():
    N, C, H, W, K, R, S, ph, pw, sh, sw, P, Q = _epi_shapes()
    x = RNG.standard_normal((N, C, H, W))
    dy = RNG.standard_normal((N, K, P, Q))
    bk, bc = RNG.standard_normal(K), RNG.standard_normal(C)
    y0, dx0 = RNG.standard_normal((N, K, P, Q)), RNG.standard_normal((N, C, H, W))
    dw0 = RNG.standard_normal((K, C, R, S))
    wz = np.zeros((K, C, R, S))
    y = oracle.conv2d_fwd_ex(x, wz, bk, 0.5, y0, (ph, pw), (sh, sw))
    for n, k, p, q in itertools.product(range(N), range(K), range(P), range(Q)):
        assert y[n, k, p, q] == bk[k] + 0.5 * y0[n, k, p, q]
    dx = oracle.conv2d_bwd_data_ex(dy, wz, (H, W), bc, 1.0, dx0, (ph, pw), (sh, sw))
    for n, c, h, w in itertools.product(range(N), range(C), range(H), range(W)):
        assert dx[n, c, h, w] == bc[c] + dx0[n, c, h, w]
    dw = oracle.conv2d_bwd_filter_ex(x, np.zeros((N, K, P, Q)), (R, S), 2.0, dw0, (ph, pw), (sh, sw))
    assert np.array_equal(dw, 2.0 * dw0)
    # beta = 0 never reads the old value (NaN there must not leak)
    nan_old = np.full((N, K, P, Q), np.nan)
    assert np.all(np.isfinite(oracle.conv2d_fwd_ex(x, wz, bk, 0.0, nan_old, (ph, pw), (sh, sw))))


def _chan_sum_pins(chan_sum):
    """Closed forms for a per-channel sum over (n, h, w); True if all hold."""
    ok = True
    N, Ch, Hh, Ww = 3, 4, 2, 5
    HW = Hh * Ww
    t = np.arange(N * Ch * HW, dtype=np.float64).reshape(N, Ch, Hh, Ww)
    # t[n, ch, i] = (n*Ch + ch)*HW + i, so the sum over n < N, i < HW is
    # HW^2 * (Ch*N*(N-1)/2 + ch*N) + N*HW*(HW-1)/2
    want = np.array([HW * HW * (Ch * N * (N - 1) / 2 + ch * N) + N * HW * (HW - 1) / 2 for ch in range(Ch)])
    got = chan_sum(t)
    ok &= got.shape == (Ch,) and bool(np.array_equal(got, want))
    ok &= bool(np.array_equal(chan_sum(np.full((N, Ch, Hh, Ww), 0.25)), np.full(Ch, 0.25 * N * HW)))
    return ok


def test_channel_sum_closed_forms():
    assert _chan_sum_pins(oracle.channel_sum)
    old = RNG.standard_normal(4)
    t = RNG.standard_normal((2, 4, 3, 3))
    assert np.allclose(oracle.channel_sum(t, 1.0, old), t.sum(axis=(0, 2, 3)) + old, rtol=0, atol=1e-12)


@pytest.mark.parametrize("mistake", ["drop_batch", "wrong_axis", "drop_last_row"])
def test_channel_sum_pins_catch_planted_mistakes(mistake):
    def bad(t):
        if mistake == "drop_batch":
            return t[0].sum(axis=(1, 2))
        if mistake == "wrong_axis":
            return t.sum(axis=(1, 2, 3))
        return t[:, :, :-1, :].sum(axis=(0, 2, 3))
    assert not _chan_sum_pins(bad)


def test_bias_gradient_is_derivative_of_bias():
    """<conv_ex(x, w, b), dy> is affine in b with slope channel_sum(dy) (convolution bias), and
    <bwd_data_ex(dy, w, b), g> has slope channel_sum(g) (deconvolution bias, g = its output
    gradient): finite differences of size 1 are exact in fp64 up to rounding."""
    N, C, H, W, K, R, S, ph, pw, sh, sw, P, Q = _epi_shapes()
    x = RNG.standard_normal((N, C, H, W))
    w = RNG.standard_normal((K, C, R, S))
    dy = RNG.standard_normal((N, K, P, Q))
    g = RNG.standard_normal((N, C, H, W))
    bk, bc = RNG.standard_normal(K), RNG.standard_normal(C)
    base = np.vdot(oracle.conv2d_fwd_ex(x, w, bk, 0.0, None, (ph, pw), (sh, sw)), dy)
    db = oracle.channel_sum(dy)
    for k in range(K):
        e = bk.copy()
        e[k] += 1.0
        slope = np.vdot(oracle.conv2d_fwd_ex(x, w, e, 0.0, None, (ph, pw), (sh, sw)), dy) - base
        assert abs(slope - db[k]) <= 1e-9 * max(1.0, abs(db[k]))
    base = np.vdot(oracle.conv2d_bwd_data_ex(dy, w, (H, W), bc, 0.0, None, (ph, pw), (sh, sw)), g)
    dbc = oracle.channel_sum(g)
    for c in range(C):
        e = bc.copy()
        e[c] += 1.0
        slope = np.vdot(oracle.conv2d_bwd_data_ex(dy, w, (H, W), e, 0.0, None, (ph, pw), (sh, sw)), g) - base
        assert abs(slope - dbc[c]) <= 1e-9 * max(1.0, abs(dbc[c]))


def test_epilogue_torch_cpu_fp64_witness():
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    N, C, H, W, K, R, S, ph, pw, sh, sw, P, Q = _epi_shapes()
    x = RNG.standard_normal((N, C, H, W))
    w = RNG.standard_normal((K, C, R, S))
    dy = RNG.standard_normal((N, K, P, Q))
    bk, bc = RNG.standard_normal(K), RNG.standard_normal(C)
    y_ref = F.conv2d(torch.from_numpy(x), torch.from_numpy(w), torch.from_numpy(bk), stride=(sh, sw),
                     padding=(ph, pw)).numpy()
    y = oracle.conv2d_fwd_ex(x, w, bk, 0.0, None, (ph, pw), (sh, sw))
    assert np.max(np.abs(y - y_ref)) <= 1e-12 * max(1.0, np.max(np.abs(y_ref)))
    # deconvolution with bias: conv_transpose2d(dy, w as (in=K, out=C), bias over C)
    outpad = (H - ((P - 1) * sh - 2 * ph + R), W - ((Q - 1) * sw - 2 * pw + S))
    d_ref = F.conv_transpose2d(torch.from_numpy(dy), torch.from_numpy(w), torch.from_numpy(bc),
                               stride=(sh, sw), padding=(ph, pw), output_padding=outpad).numpy()
    d = oracle.conv2d_bwd_data_ex(dy, w, (H, W), bc, 0.0, None, (ph, pw), (sh, sw))
    assert np.max(np.abs(d - d_ref)) <= 1e-12 * max(1.0, np.max(np.abs(d_ref)))


# --------------------------------------------------------------------------- convolution mode
# cuDNN's convolution mode (the SystemDS page picks CUDNN_CROSS_CORRELATION, the other value
# of the same descriptor field): the filter enters rotated by 180 degrees.

def test_convolution_mode_torch_witness():
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    N, C, H, W, K, R, S, ph, pw, sh, sw, P, Q = _epi_shapes()
    x = RNG.standard_normal((N, C, H, W))
    w = RNG.standard_normal((K, C, R, S))
    ref = F.conv2d(torch.from_numpy(x), torch.from_numpy(w).flip(2, 3), stride=(sh, sw), padding=(ph, pw)).numpy()
    got = oracle.conv2d_fwd_ex(x, w, None, 0.0, None, (ph, pw), (sh, sw), flip=True)
    assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))
    # a half flip (rows only) is not the same op: the witness separates them
    half = oracle.conv2d_fwd(x, np.ascontiguousarray(w[:, :, ::-1, :]), (ph, pw), (sh, sw))
    assert np.max(np.abs(half - ref)) > 1e-6


def test_convolution_mode_adjoint_identities():
    """<fwd(x, w), dy> = <x, bwd_data(dy, w)> = <w, bwd_filter(x, dy)> in convolution mode
    too: ties the three flipped ops together (a flip missing or misplaced in one of them
    breaks an equality)."""
    for case in ADJ_CASES[:3]:
        N, C, H, W, K, R, S, ph, pw, sh, sw = case
        P, Q = oracle.output_dim(H, ph, R, sh), oracle.output_dim(W, pw, S, sw)
        x = RNG.standard_normal((N, C, H, W))
        w = RNG.standard_normal((K, C, R, S))
        dy = RNG.standard_normal((N, K, P, Q))
        a = np.vdot(oracle.conv2d_fwd_ex(x, w, None, 0.0, None, (ph, pw), (sh, sw), flip=True), dy)
        b = np.vdot(x, oracle.conv2d_bwd_data_ex(dy, w, (H, W), None, 0.0, None, (ph, pw), (sh, sw), flip=True))
        c = np.vdot(w, oracle.conv2d_bwd_filter_ex(x, dy, (R, S), 0.0, None, (ph, pw), (sh, sw), flip=True))
        assert abs(a - b) <= 1e-10 * max(1.0, abs(a)) and abs(a - c) <= 1e-10 * max(1.0, abs(a))
        if R * S > 1:
            # the unflipped filter gradient does not satisfy the flipped identity
            c0 = np.vdot(w, oracle.conv2d_bwd_filter(x, dy, (R, S), (ph, pw), (sh, sw)))
            assert abs(a - c0) > 1e-8 * max(1.0, abs(a))


# --------------------------------------------------------------------------- dilation
# cuDNN's convolution-descriptor dilation (set to 1, 1 on the SystemDS page): tap (r, s) reads
# the window at (r*dh, s*dw).  Pinned by PyTorch CPU fp64 for all three ops and by the adjoint
# identities.
DIL_CASES = [
    ((2, 3, 12, 13, 4, 3, 3, 2, 2, 1, 1), (2, 2)),
    ((1, 2, 17, 15, 3, 3, 2, 2, 1, 2, 1), (2, 3)),
    ((2, 4, 11, 16, 5, 2, 3, 1, 2, 1, 2), (3, 2)),
]


def _dil_out(H, W, R, S, ph, pw, sh, sw, dil):
    dh, dw = dil
    return oracle.output_dim(H, ph, dh * (R - 1) + 1, sh), oracle.output_dim(W, pw, dw * (S - 1) + 1, sw)


@pytest.mark.parametrize("case,dil", DIL_CASES)
def test_dilation_torch_witness(case, dil):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    N, C, H, W, K, R, S, ph, pw, sh, sw = case
    P, Q = _dil_out(H, W, R, S, ph, pw, sh, sw, dil)
    x = RNG.standard_normal((N, C, H, W))
    w = RNG.standard_normal((K, C, R, S))
    dy = RNG.standard_normal((N, K, P, Q))
    tx, tw, tdy = (torch.from_numpy(a) for a in (x, w, dy))
    kw = dict(stride=(sh, sw), padding=(ph, pw), dilation=dil)
    refs = (F.conv2d(tx, tw, **kw).numpy(),
            torch.nn.grad.conv2d_input((N, C, H, W), tw, tdy, **kw).numpy(),
            torch.nn.grad.conv2d_weight(tx, (K, C, R, S), tdy, **kw).numpy())
    gots = (oracle.conv2d_fwd_ex(x, w, None, 0.0, None, (ph, pw), (sh, sw), dilation=dil),
            oracle.conv2d_bwd_data_ex(dy, w, (H, W), None, 0.0, None, (ph, pw), (sh, sw), dilation=dil),
            oracle.conv2d_bwd_filter_ex(x, dy, (R, S), 0.0, None, (ph, pw), (sh, sw), dilation=dil))
    for got, ref in zip(gots, refs):
        assert got.shape == ref.shape
        assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


@pytest.mark.parametrize("case,dil", DIL_CASES)
def test_dilation_adjoint_identities(case, dil):
    N, C, H, W, K, R, S, ph, pw, sh, sw = case
    P, Q = _dil_out(H, W, R, S, ph, pw, sh, sw, dil)
    x = RNG.standard_normal((N, C, H, W))
    w = RNG.standard_normal((K, C, R, S))
    dy = RNG.standard_normal((N, K, P, Q))
    for flip in (False, True):
        a = np.vdot(oracle.conv2d_fwd_ex(x, w, None, 0.0, None, (ph, pw), (sh, sw), flip, dil), dy)
        b = np.vdot(x, oracle.conv2d_bwd_data_ex(dy, w, (H, W), None, 0.0, None, (ph, pw), (sh, sw), flip, dil))
        c = np.vdot(w, oracle.conv2d_bwd_filter_ex(x, dy, (R, S), 0.0, None, (ph, pw), (sh, sw), flip, dil))
        assert abs(a - b) <= 1e-10 * max(1.0, abs(a)) and abs(a - c) <= 1e-10 * max(1.0, abs(a))


# --------------------------------------------------------------------------- groups
# cuDNN's group count of the convolution descriptor: `groups` independent convolutions on
# channel slices, filter K x C/groups x R x S.  Pinned by PyTorch CPU fp64 (groups=) for the
# three ops, with dilation and convolution mode mixed in, and by the adjoint identities.
GROUP_CASES = [
    ((2, 6, 9, 10, 9, 3, 3, 1, 1, 1, 1), 3, (1, 1)),
    ((1, 8, 11, 12, 8, 3, 2, 1, 0, 2, 1), 8, (1, 1)),    # depthwise
    ((2, 4, 13, 11, 6, 3, 3, 2, 2, 1, 2), 2, (2, 1)),
]


@pytest.mark.parametrize("case,groups,dil", GROUP_CASES)
def test_groups_torch_witness(case, groups, dil):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    N, C, H, W, K, R, S, ph, pw, sh, sw = case
    P, Q = _dil_out(H, W, R, S, ph, pw, sh, sw, dil)
    x = RNG.standard_normal((N, C, H, W))
    w = RNG.standard_normal((K, C // groups, R, S))
    dy = RNG.standard_normal((N, K, P, Q))
    tx, tw, tdy = (torch.from_numpy(a) for a in (x, w, dy))
    kw = dict(stride=(sh, sw), padding=(ph, pw), dilation=dil, groups=groups)
    refs = (F.conv2d(tx, tw, **kw).numpy(),
            torch.nn.grad.conv2d_input((N, C, H, W), tw, tdy, **kw).numpy(),
            torch.nn.grad.conv2d_weight(tx, (K, C // groups, R, S), tdy, **kw).numpy())
    gots = (oracle.conv2d_fwd_ex(x, w, None, 0.0, None, (ph, pw), (sh, sw), dilation=dil, groups=groups),
            oracle.conv2d_bwd_data_ex(dy, w, (H, W), None, 0.0, None, (ph, pw), (sh, sw), dilation=dil, groups=groups),
            oracle.conv2d_bwd_filter_ex(x, dy, (R, S), 0.0, None, (ph, pw), (sh, sw), dilation=dil, groups=groups))
    for got, ref in zip(gots, refs):
        assert got.shape == ref.shape
        assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


@pytest.mark.parametrize("case,groups,dil", GROUP_CASES)
def test_groups_adjoint_identities(case, groups, dil):
    N, C, H, W, K, R, S, ph, pw, sh, sw = case
    P, Q = _dil_out(H, W, R, S, ph, pw, sh, sw, dil)
    x = RNG.standard_normal((N, C, H, W))
    w = RNG.standard_normal((K, C // groups, R, S))
    dy = RNG.standard_normal((N, K, P, Q))
    for flip in (False, True):
        a = np.vdot(oracle.conv2d_fwd_ex(x, w, None, 0.0, None, (ph, pw), (sh, sw), flip, dil, groups), dy)
        b = np.vdot(x, oracle.conv2d_bwd_data_ex(dy, w, (H, W), None, 0.0, None, (ph, pw), (sh, sw), flip, dil, groups))
        c = np.vdot(w, oracle.conv2d_bwd_filter_ex(x, dy, (R, S), 0.0, None, (ph, pw), (sh, sw), flip, dil, groups))
        assert abs(a - b) <= 1e-10 * max(1.0, abs(a)) and abs(a - c) <= 1e-10 * max(1.0, abs(a))

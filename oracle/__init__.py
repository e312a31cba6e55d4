"""fp64 CPU oracle for NCHW conv2d (and NCDHW conv3d) -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (``convolution_nchw_conv2d_gb300``)
never imports it and shares no code with it.

The convolution arithmetic lives in ``conv2d_oracle.c`` and ``conv3d_oracle.c``
(plain C, fp64, gather form, OpenMP over output elements); this module compiles
them with gcc into one library and marshals numpy arrays through ctypes.  The fused epilogues (bias, beta) and the per-channel
bias-gradient sums are written here directly in fp64 numpy on top of those ops.
Inputs of any float dtype are widened exactly to fp64 before the call.

Citations (page titles): Apache SystemDS ``LibMatrixCuDNNConvolutionAlgorithm.java``
(descriptor integers, NCHW / KCRS layouts, cross-correlation, dilation 1);
Apache MXNet ``mkldnn_deconvolution.cc`` (deconvolution forward = convolution
backward-data with the weight's in/out channel roles swapped); the C#
``FilterDescriptor.SetFilter4dDescriptor`` examples (overwrite, alpha = 1,
beta = 0).

Parity status: all functions pinned by ``tests/test_oracle_pins.py`` (2-D) and
``tests/test_oracle_pins_3d.py`` (3-D); NaN/Inf propagation is parity unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "conv2d_oracle.c"), os.path.join(_HERE, "conv3d_oracle.c")]
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle_conv2d.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2 -fopenmp) into ``oracle/_build``."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(map(os.path.getmtime, _SRCS)):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
                               "-o", tmp] + _SRCS)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    """Set the ctypes signatures of the oracle library's entry points; returns lib."""
    i = ctypes.c_int
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    lib.oracle_output_dim.argtypes = [i, i, i, i]
    lib.oracle_output_dim.restype = i
    for name in ("oracle_conv2d_fwd", "oracle_conv2d_bwd_data", "oracle_conv2d_bwd_filter"):
        getattr(lib, name).argtypes = [dp, dp, dp] + [i] * 13
        getattr(lib, name).restype = None
    lib.oracle_deconv2d_fwd_scatter.argtypes = [dp, dp, dp] + [i] * 13
    lib.oracle_deconv2d_fwd_scatter.restype = None
    for name in ("oracle_conv2d_fwd_at", "oracle_conv2d_bwd_data_at",
                 "oracle_conv2d_bwd_filter_at"):
        getattr(lib, name).argtypes = [dp, dp] + [i] * 13 + [ip, i64, dp]
        getattr(lib, name).restype = None
    ivp = ctypes.POINTER(ctypes.c_int)
    for name in ("oracle_conv3d_fwd", "oracle_conv3d_bwd_data", "oracle_conv3d_bwd_filter"):
        getattr(lib, name).argtypes = [dp, dp, dp, ivp]
        getattr(lib, name).restype = None
    for name in ("oracle_conv3d_fwd_at", "oracle_conv3d_bwd_data_at", "oracle_conv3d_bwd_filter_at"):
        getattr(lib, name).argtypes = [dp, dp, ivp, ip, i64, dp]
        getattr(lib, name).restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _f64(a) -> np.ndarray:
    """Exact widening to a C-contiguous fp64 numpy array (torch tensors accepted)."""
    if hasattr(a, "detach"):
        a = a.detach().cpu().float().numpy() if str(a.dtype) == "torch.bfloat16" else a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def output_dim(inp: int, pad: int, k: int, stride: int) -> int:
    """floor((inp + 2*pad - k)/stride) + 1, 0 if the window never fits, -1 on bad input."""
    return _load().oracle_output_dim(inp, pad, k, stride)


def _geom(x_shape, w_shape, pad, stride):
    N, C, H, W = x_shape
    K, C2, R, S = w_shape
    assert C == C2, "channel mismatch between x and w"
    ph, pw = pad
    sh, sw = stride
    P = output_dim(H, ph, R, sh)
    Q = output_dim(W, pw, S, sw)
    return N, C, H, W, K, R, S, ph, pw, sh, sw, P, Q


def _pair(v):
    return (v, v) if isinstance(v, int) else tuple(v)


def conv2d_fwd(x, w, pad=0, stride=1) -> np.ndarray:
    """y = cross-correlation of zero-padded x with w (NCHW, KCRS) in fp64."""
    x, w = _f64(x), _f64(w)
    g = _geom(x.shape, w.shape, _pair(pad), _pair(stride))
    N, C, H, W, K, R, S, ph, pw, sh, sw, P, Q = g
    y = np.empty((N, K, P, Q), dtype=np.float64)
    _load().oracle_conv2d_fwd(_ptr(x), _ptr(w), _ptr(y), *g)
    return y


def conv2d_bwd_data(dy, w, x_hw, pad=0, stride=1) -> np.ndarray:
    """dx (N,C,H,W) from dy (N,K,P,Q) and w (K,C,R,S); x_hw = (H, W) is explicit
    because for stride > 1 several H give the same P."""
    dy, w = _f64(dy), _f64(w)
    N, K, P, Q = dy.shape
    K2, C, R, S = w.shape
    assert K == K2
    H, W = x_hw
    ph, pw = _pair(pad)
    sh, sw = _pair(stride)
    assert output_dim(H, ph, R, sh) == P and output_dim(W, pw, S, sw) == Q, "P/Q mismatch"
    dx = np.empty((N, C, H, W), dtype=np.float64)
    _load().oracle_conv2d_bwd_data(_ptr(dy), _ptr(w), _ptr(dx),
                                   N, C, H, W, K, R, S, ph, pw, sh, sw, P, Q)
    return dx


def conv2d_bwd_filter(x, dy, rs, pad=0, stride=1) -> np.ndarray:
    """dw (K,C,R,S) from x (N,C,H,W) and dy (N,K,P,Q); rs = (R, S)."""
    x, dy = _f64(x), _f64(dy)
    N, C, H, W = x.shape
    N2, K, P, Q = dy.shape
    assert N == N2
    R, S = rs
    ph, pw = _pair(pad)
    sh, sw = _pair(stride)
    assert output_dim(H, ph, R, sh) == P and output_dim(W, pw, S, sw) == Q, "P/Q mismatch"
    dw = np.empty((K, C, R, S), dtype=np.float64)
    _load().oracle_conv2d_bwd_filter(_ptr(x), _ptr(dy), _ptr(dw),
                                     N, C, H, W, K, R, S, ph, pw, sh, sw, P, Q)
    return dw


def deconv2d_fwd_scatter(inp, wt, out_hw, pad=0, stride=1) -> np.ndarray:
    """Transposed convolution by scatter: inp (N,Ci,Hi,Wi), wt (Ci,Co,R,S) -> (N,Co,Ho,Wo)."""
    inp, wt = _f64(inp), _f64(wt)
    N, Ci, Hi, Wi = inp.shape
    Ci2, Co, R, S = wt.shape
    assert Ci == Ci2
    Ho, Wo = out_hw
    ph, pw = _pair(pad)
    sh, sw = _pair(stride)
    out = np.empty((N, Co, Ho, Wo), dtype=np.float64)
    _load().oracle_deconv2d_fwd_scatter(_ptr(inp), _ptr(wt), _ptr(out),
                                        N, Ci, Hi, Wi, Co, R, S, ph, pw, sh, sw, Ho, Wo)
    return out


# ------------------------------------------------------------------ fused epilogues
# Page "mkldnn_deconvolution.cc": the deconvolution forward adds an optional bias per output
# channel and either writes or adds to its output (MKLDNNDeconvFwd::Execute, OutMem(req));
# its backward-weights pass also yields the bias gradient (ScheduleBwdWeights, BiasGradMem).
# The rule for every output element is  D + bias[channel] + beta * old  (beta 0 writes,
# beta 1 adds), written out below on top of the plain ops, in fp64.

def _epilogue(d, bias, beta, old, channel_axis):
    out = np.array(d, dtype=np.float64, copy=True)
    if bias is not None:
        b = _f64(bias).reshape(-1)
        shape = [1] * out.ndim
        shape[channel_axis] = b.shape[0]
        out = out + b.reshape(shape)
    if beta != 0.0:
        out = out + float(beta) * _f64(old)
    return out


# Convolution mode (cuDNN's CUDNN_CONVOLUTION, the alternative to the CUDNN_CROSS_CORRELATION
# the SystemDS page selects): the filter enters rotated by 180 degrees, w[k,c,R-1-r,S-1-s]; the
# filter gradient of that op is the cross-correlation gradient rotated back.

def _rot180(w):
    return np.ascontiguousarray(_f64(w)[:, :, ::-1, ::-1])


# Dilation (cuDNN's convolution-descriptor dilation, which the SystemDS page sets to 1, 1):
# tap (r, s) reads the input at offset (r*dh, s*dw) of the window.  That is the undilated op
# with the zero-inserted filter of extent (dh*(R-1)+1, dw*(S-1)+1) holding w[r, s] at
# (r*dh, s*dw); the filter gradient is that op's gradient read back at those places.

def dilate_filter(w, dilation) -> np.ndarray:
    dh, dw = _pair(dilation)
    w = _f64(w)
    K, C, R, S = w.shape
    out = np.zeros((K, C, dh * (R - 1) + 1, dw * (S - 1) + 1))
    out[:, :, ::dh, ::dw] = w
    return out


# Groups (cuDNN's group count of the convolution descriptor): the C input and K output
# channels split into `groups` independent convolutions, group g taking input channels
# g*C/groups .. and output channels g*K/groups .. with filter rows g*K/groups .. of a
# K x C/groups x R x S filter.  Written out as one plain op per group on channel slices.

def conv2d_fwd_ex(x, w, bias=None, beta=0.0, y_old=None, pad=0, stride=1, flip=False, dilation=1,
                  groups=1) -> np.ndarray:
    """y = conv(x, w) + bias[k] + beta * y_old (bias per output channel k, axis 1 of y); flip:
    convolution mode; dilation, groups: see above."""
    x = _f64(x)
    wf = dilate_filter(_rot180(w) if flip else w, dilation)
    Cg, Kg = x.shape[1] // groups, wf.shape[0] // groups
    y = np.concatenate([conv2d_fwd(x[:, g * Cg:(g + 1) * Cg], wf[g * Kg:(g + 1) * Kg], pad, stride)
                        for g in range(groups)], axis=1)
    return _epilogue(y, bias, beta, y_old, 1)


def conv2d_bwd_data_ex(dy, w, x_hw, bias=None, beta=0.0, dx_old=None, pad=0, stride=1, flip=False,
                       dilation=1, groups=1) -> np.ndarray:
    """dx = bwd_data(dy, w) + bias[c] + beta * dx_old (bias per channel c of dx: the bias of
    the deconvolution whose output dx is); flip: convolution mode; dilation, groups: see above."""
    dy = _f64(dy)
    wf = dilate_filter(_rot180(w) if flip else w, dilation)
    Kg = dy.shape[1] // groups
    dx = np.concatenate([conv2d_bwd_data(dy[:, g * Kg:(g + 1) * Kg], wf[g * Kg:(g + 1) * Kg], x_hw, pad, stride)
                         for g in range(groups)], axis=1)
    return _epilogue(dx, bias, beta, dx_old, 1)


def conv2d_bwd_filter_ex(x, dy, rs, beta=0.0, dw_old=None, pad=0, stride=1, flip=False, dilation=1,
                         groups=1) -> np.ndarray:
    """dw (K, C/groups, R, S) = bwd_filter(x, dy) + beta * dw_old; flip: the gradient of the
    rotated filter; dilation, groups: see above."""
    x, dy = _f64(x), _f64(dy)
    dh, dwl = _pair(dilation)
    R, S = rs
    Cg, Kg = x.shape[1] // groups, dy.shape[1] // groups
    big = np.concatenate([conv2d_bwd_filter(x[:, g * Cg:(g + 1) * Cg], dy[:, g * Kg:(g + 1) * Kg],
                                            (dh * (R - 1) + 1, dwl * (S - 1) + 1), pad, stride)
                          for g in range(groups)], axis=0)
    dw = np.ascontiguousarray(big[:, :, ::dh, ::dwl])
    return _epilogue(_rot180(dw) if flip else dw, None, beta, dw_old, 0)


def channel_sum(t, beta=0.0, old=None) -> np.ndarray:
    """out[ch] = sum over images and pixels of t[n, ch, :, :] (+ beta * old[ch]) in fp64: the
    convolution bias gradient for t = dy, the deconvolution bias gradient for t = its output
    gradient."""
    t = _f64(t)
    out = t.sum(axis=(0, 2, 3))
    if beta != 0.0:
        out = out + float(beta) * _f64(old)
    return out


def _at(fn, a, b, dims, idx):
    a, b = _f64(a), _f64(b)
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64))
    out = np.empty(idx.shape[0], dtype=np.float64)
    fn(_ptr(a), _ptr(b), *dims,
       idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), ctypes.c_int64(idx.shape[0]), _ptr(out))
    return out


def conv2d_fwd_at(x, w, dims, idx) -> np.ndarray:
    """Forward outputs at flat (n,k,p,q) indices; dims = the 13 descriptor ints."""
    return _at(_load().oracle_conv2d_fwd_at, x, w, dims, idx)


def conv2d_bwd_data_at(dy, w, dims, idx) -> np.ndarray:
    """Backward-data outputs at flat (n,c,h,w) indices."""
    return _at(_load().oracle_conv2d_bwd_data_at, dy, w, dims, idx)


def conv2d_bwd_filter_at(x, dy, dims, idx) -> np.ndarray:
    """Backward-filter outputs at flat (k,c,r,s) indices."""
    return _at(_load().oracle_conv2d_bwd_filter_at, x, dy, dims, idx)


# ------------------------------------------------------------------ 3-D (NCDHW)
# Page "mkldnn_deconvolution.cc" (Apache MXNet): SupportMKLDNNDeconv accepts kernels of one to
# three spatial dims on an input with two more dims, and DeconvDescCreator takes one stride /
# pad / dilation per spatial dim (equal counts, 1 to 3).  The 3-D ops below take
# x (N,C,D,H,W), w (K,C/groups,T,R,S), y / dy (N,K,Z,P,Q); groups split the channels as in
# the 2-D ops.  The per-element definitions are in conv3d_oracle.c.

def _triple(v):
    return (v, v, v) if isinstance(v, int) else tuple(v)


def output_dim_dilated(inp: int, pad: int, k: int, stride: int, dil: int) -> int:
    """Output extent along one dim for a filter of k taps dilated by dil (extent dil*(k-1)+1)."""
    return output_dim(inp, pad, dil * (k - 1) + 1, stride)


def _dims3(N, C, DHW, K, TRS, pad, stride, dilation):
    pads, strides, dils = _triple(pad), _triple(stride), _triple(dilation)
    out = [output_dim_dilated(i, p_, k, s_, d_) for i, p_, k, s_, d_ in zip(DHW, pads, TRS, strides, dils)]
    dims = [N, C, *DHW, K, *TRS, *pads, *strides, *dils, *out]
    return np.ascontiguousarray(np.asarray(dims, dtype=np.int32)), tuple(out)


def _iptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def conv3d_fwd(x, w, pad=0, stride=1, dilation=1, groups=1) -> np.ndarray:
    """y (N,K,Z,P,Q) = cross-correlation of zero-padded x (N,C,D,H,W) with w (K,C/groups,T,R,S)."""
    x, w = _f64(x), _f64(w)
    N, C = x.shape[:2]
    K, Cg = w.shape[:2]
    assert C == Cg * groups and K % groups == 0, "channel / group mismatch"
    Kg = K // groups
    parts = []
    for g in range(groups):
        xs = np.ascontiguousarray(x[:, g * Cg:(g + 1) * Cg])
        ws = np.ascontiguousarray(w[g * Kg:(g + 1) * Kg])
        dims, (Z, P, Q) = _dims3(N, Cg, x.shape[2:], Kg, w.shape[2:], pad, stride, dilation)
        y = np.empty((N, Kg, Z, P, Q), dtype=np.float64)
        _load().oracle_conv3d_fwd(_ptr(xs), _ptr(ws), _ptr(y), _iptr(dims))
        parts.append(y)
    return np.concatenate(parts, axis=1)


def conv3d_bwd_data(dy, w, x_dhw, pad=0, stride=1, dilation=1, groups=1) -> np.ndarray:
    """dx (N,C,D,H,W) from dy (N,K,Z,P,Q) and w (K,C/groups,T,R,S); x_dhw = (D, H, W)."""
    dy, w = _f64(dy), _f64(w)
    N, K = dy.shape[:2]
    K2, Cg = w.shape[:2]
    assert K == K2 and K % groups == 0
    Kg = K // groups
    parts = []
    for g in range(groups):
        dys = np.ascontiguousarray(dy[:, g * Kg:(g + 1) * Kg])
        ws = np.ascontiguousarray(w[g * Kg:(g + 1) * Kg])
        dims, out = _dims3(N, Cg, tuple(x_dhw), Kg, w.shape[2:], pad, stride, dilation)
        assert out == tuple(dy.shape[2:]), "Z/P/Q mismatch"
        dx = np.empty((N, Cg, *x_dhw), dtype=np.float64)
        _load().oracle_conv3d_bwd_data(_ptr(dys), _ptr(ws), _ptr(dx), _iptr(dims))
        parts.append(dx)
    return np.concatenate(parts, axis=1)


def conv3d_bwd_filter(x, dy, trs, pad=0, stride=1, dilation=1, groups=1) -> np.ndarray:
    """dw (K,C/groups,T,R,S) from x (N,C,D,H,W) and dy (N,K,Z,P,Q); trs = (T, R, S)."""
    x, dy = _f64(x), _f64(dy)
    N, C = x.shape[:2]
    N2, K = dy.shape[:2]
    assert N == N2 and C % groups == 0 and K % groups == 0
    Cg, Kg = C // groups, K // groups
    parts = []
    for g in range(groups):
        xs = np.ascontiguousarray(x[:, g * Cg:(g + 1) * Cg])
        dys = np.ascontiguousarray(dy[:, g * Kg:(g + 1) * Kg])
        dims, out = _dims3(N, Cg, x.shape[2:], Kg, tuple(trs), pad, stride, dilation)
        assert out == tuple(dy.shape[2:]), "Z/P/Q mismatch"
        dw = np.empty((Kg, Cg, *trs), dtype=np.float64)
        _load().oracle_conv3d_bwd_filter(_ptr(xs), _ptr(dys), _ptr(dw), _iptr(dims))
        parts.append(dw)
    return np.concatenate(parts, axis=0)


def _at3(fn, a, b, dims, idx):
    a, b = _f64(a), _f64(b)
    dims = np.ascontiguousarray(np.asarray(dims, dtype=np.int32))
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64))
    out = np.empty(idx.shape[0], dtype=np.float64)
    fn(_ptr(a), _ptr(b), _iptr(dims), idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
       ctypes.c_int64(idx.shape[0]), _ptr(out))
    return out


def conv3d_dims(x_shape, w_shape, pad=0, stride=1, dilation=1):
    """The 21 descriptor ints of the C 3-D ops for x (N,C,D,H,W) and w (K,C,T,R,S), one group."""
    dims, _ = _dims3(x_shape[0], x_shape[1], tuple(x_shape[2:]), w_shape[0], tuple(w_shape[2:]), pad, stride,
                     dilation)
    return dims


def conv3d_fwd_at(x, w, dims, idx) -> np.ndarray:
    """Forward outputs at flat (n,k,z,p,q) indices; dims from conv3d_dims (one group)."""
    return _at3(_load().oracle_conv3d_fwd_at, x, w, dims, idx)


def conv3d_bwd_data_at(dy, w, dims, idx) -> np.ndarray:
    """Backward-data outputs at flat (n,c,z,h,w) indices."""
    return _at3(_load().oracle_conv3d_bwd_data_at, dy, w, dims, idx)


def conv3d_bwd_filter_at(x, dy, dims, idx) -> np.ndarray:
    """Backward-filter outputs at flat (k,c,t,r,s) indices."""
    return _at3(_load().oracle_conv3d_bwd_filter_at, x, dy, dims, idx)


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return _load().oracle_num_threads()

"""GB300 (sm_103a) NCHW 2-D convolution: forward, backward-data, backward-filter.

A thin ctypes binding over ``libconv2d_gb300.so`` (C ABI in
``include/conv2d_gb300.h``).  The functions here only marshal torch tensors
(device memory and the current CUDA stream) into the C calls; every step of
the computation runs in the library's CUDA kernels.  If the library is missing
or cannot be loaded, every call raises -- there is no fallback path.

Names follow the descriptor of the Apache SystemDS cuDNN wrapper page
(``LibMatrixCuDNNConvolutionAlgorithm.java``): N, C, H, W, K, R, S, pad_h, pad_w,
stride_h, stride_w, P, Q.  ``deconv2d_fwd`` maps transposed convolution onto
backward-data with the weight read as (deconv_in, deconv_out, R, S) (Apache MXNet
``mkldnn_deconvolution.cc``, MKLDNNDeconvFwd::Execute comment).
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "conv2d_fwd", "conv2d_bwd_data", "conv2d_bwd_filter", "deconv2d_fwd", "conv2d_fwd_noalloc",
    "conv1d_fwd", "conv1d_bwd_data", "conv1d_bwd_filter", "MODE_CROSS_CORRELATION", "MODE_CONVOLUTION",
    "conv2d_workspace_size", "conv2d_output_dim", "conv2d_device_status", "conv2d_strerror",
    "conv2d_kernel_launches", "conv2d_bwd", "conv3d_fwd", "conv3d_bwd_data", "conv3d_bwd_filter",
    "Conv2dError", "lib_path", "load_library", "OP_FWD", "OP_BWD_DATA", "OP_BWD_FILTER", "OP_BWD",
    "DTYPE_F32", "DTYPE_BF16",
]

OP_FWD, OP_BWD_DATA, OP_BWD_FILTER, OP_BWD = 0, 1, 2, 3
MODE_CROSS_CORRELATION, MODE_CONVOLUTION = 0, 1
DTYPE_F32, DTYPE_BF16 = 0, 1

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libconv2d_gb300.so")
_lib = None
_lock = threading.Lock()


class Conv2dError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {conv2d_strerror(code)} (code {code})")


def lib_path() -> str:
    return _LIB_PATH


EXPORTS = ("conv2d_output_dim", "conv2d_workspace_size", "conv2d_workspace_size_ex", "conv2d_fwd", "conv2d_bwd_data",
           "conv2d_bwd_filter", "conv2d_fwd_ex", "conv2d_bwd_data_ex", "conv2d_bwd_filter_ex",
           "conv2d_fwd_noalloc", "conv2d_device_status", "conv2d_strerror", "conv2d_kernel_launches",
           "conv3d_workspace_size", "conv3d_fwd", "conv3d_bwd_data", "conv3d_bwd_filter", "conv2d_bwd")


def load_library():
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(_LIB_PATH)
        i, sz, vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
        lib.conv2d_output_dim.argtypes = [i, i, i, i, ctypes.POINTER(i)]
        lib.conv2d_output_dim.restype = i
        lib.conv2d_workspace_size.argtypes = [i] + [i] * 13 + [i, ctypes.POINTER(sz)]
        lib.conv2d_workspace_size.restype = i
        for name in ("conv2d_fwd", "conv2d_bwd_data", "conv2d_bwd_filter"):
            f = getattr(lib, name)
            f.argtypes = [i] * 13 + [i, vp, vp, vp, vp, sz, vp]
            f.restype = i
        fl = ctypes.c_float
        for name in ("conv2d_fwd_ex", "conv2d_bwd_data_ex"):
            f = getattr(lib, name)
            f.argtypes = [i] * 16 + [i, i, vp, vp, vp, fl, vp, vp, sz, vp]
            f.restype = i
        lib.conv2d_bwd_filter_ex.argtypes = [i] * 16 + [i, i, vp, vp, fl, vp, vp, vp, vp, sz, vp]
        lib.conv2d_workspace_size_ex.argtypes = [i] + [i] * 16 + [i, ctypes.POINTER(sz)]
        lib.conv2d_workspace_size_ex.restype = i
        lib.conv2d_bwd_filter_ex.restype = i
        lib.conv2d_fwd_noalloc.argtypes = [i] * 13 + [i, vp, vp, vp, vp]
        lib.conv2d_fwd_noalloc.restype = i
        lib.conv2d_device_status.argtypes = [vp]
        lib.conv2d_device_status.restype = i
        lib.conv2d_kernel_launches.argtypes = []
        lib.conv2d_kernel_launches.restype = ctypes.c_ulonglong
        lib.conv2d_strerror.argtypes = [i]
        lib.conv2d_strerror.restype = ctypes.c_char_p
        lib.conv2d_bwd.argtypes = [i] * 13 + [i, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.conv2d_bwd.restype = i
        ip = ctypes.POINTER(i)
        lib.conv3d_workspace_size.argtypes = [i, ip, i, i, ctypes.POINTER(sz)]
        lib.conv3d_workspace_size.restype = i
        for name in ("conv3d_fwd", "conv3d_bwd_data", "conv3d_bwd_filter"):
            f = getattr(lib, name)
            f.argtypes = [ip, i, i, vp, vp, vp, vp, sz, vp]
            f.restype = i
        _lib = lib
        return lib


def conv2d_strerror(code: int) -> str:
    try:
        return load_library().conv2d_strerror(code).decode()
    except Exception:  # library missing: still describe the code
        return f"error {code}"


def conv2d_output_dim(inp: int, pad: int, k: int, stride: int) -> int:
    out = ctypes.c_int(0)
    rc = load_library().conv2d_output_dim(inp, pad, k, stride, ctypes.byref(out))
    if rc:
        raise Conv2dError(rc, "conv2d_output_dim")
    return out.value


def _pair(v):
    return (int(v), int(v)) if isinstance(v, int) else (int(v[0]), int(v[1]))


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; expected float32 or bfloat16")


def conv2d_workspace_size(op: int, dims, dtype_code: int, dilation=(1, 1), groups: int = 1) -> int:
    """Workspace bytes for `op`, the 13 descriptor integers `dims`, the dilation and groups."""
    out = ctypes.c_size_t(0)
    dh, dw = _pair(dilation)
    rc = load_library().conv2d_workspace_size_ex(op, *[int(v) for v in dims], dh, dw, int(groups), dtype_code,
                                                 ctypes.byref(out))
    if rc:
        raise Conv2dError(rc, "conv2d_workspace_size")
    return out.value


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check_tensor(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (dense NCHW / KCRS)")


def _workspace(op, dims, dt, workspace, device, dilation=(1, 1), groups=1):
    import torch
    need = conv2d_workspace_size(op, dims, dt, dilation, groups)
    if need == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace too small: need {need} bytes")
    return workspace, workspace.numel() * workspace.element_size()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def _check_vec(v, n, like, name):
    if v is None:
        return
    _check_tensor(v, name)
    if v.dtype != like.dtype or v.numel() != n or v.device != like.device:
        raise ValueError(f"{name} must be a vector of {n} {like.dtype} values on {like.device}")


def _mode(flip):
    return MODE_CONVOLUTION if flip else MODE_CROSS_CORRELATION


def _call(name, dims, dt, a, b, out, workspace, op, stream, bias=None, beta=0.0, flip=False, dilation=(1, 1),
          groups=1):
    """Forward / backward-data through the fused-epilogue entry point (bias None, beta 0,
    flip False, dilation 1 and groups 1 are the plain op)."""
    ws, wsb = _workspace(op, dims, dt, workspace, out.device, dilation, groups)
    dh, dw = _pair(dilation)
    rc = getattr(load_library(), name + "_ex")(*[int(v) for v in dims], dh, dw, int(groups), dt, _mode(flip), _ptr(a),
                                               _ptr(b),
                                               _ptr(bias),
                                               ctypes.c_float(float(beta)), _ptr(out), _ptr(ws),
                                               ctypes.c_size_t(wsb), _stream_ptr(stream))
    if rc:
        raise Conv2dError(rc, name)
    return out


def _eff(k, d):
    return d * (k - 1) + 1  # extent of a dilated filter


def conv2d_fwd(x, w, pad=0, stride=1, out=None, workspace=None, stream=None, bias=None, beta=0.0, flip=False,
               dilation=1, groups=1):
    """y = conv2d(x, w) (+ bias[k]) (+ beta * y): x (N,C,H,W), w (K,C,R,S) -> y (N,K,P,Q),
    same dtype.  With beta != 0, `out` holds the values to accumulate onto.  flip=True is
    convolution mode (the filter rotated by 180 degrees); the default is cross-correlation.
    dilation (int or pair): filter tap (r, s) reads input offset (r*dil_h, s*dil_w).  groups:
    the channels split into independent convolutions; w is (K, C/groups, R, S)."""
    import torch
    _check_tensor(x, "x")
    _check_tensor(w, "w")
    N, C, H, W = x.shape
    K, C2, R, S = w.shape
    if C2 * groups != C or K % groups != 0 or w.dtype != x.dtype:
        raise ValueError("x / w channel count, groups or dtype mismatch")
    ph, pw = _pair(pad)
    sh, sw = _pair(stride)
    dh, dw = _pair(dilation)
    P, Q = conv2d_output_dim(H, ph, _eff(R, dh), sh), conv2d_output_dim(W, pw, _eff(S, dw), sw)
    if out is None:
        if beta != 0.0:
            raise ValueError("beta != 0 accumulates onto `out`, which must then be given")
        out = torch.empty((N, K, P, Q), dtype=x.dtype, device=x.device)
    _check_vec(bias, K, x, "bias")
    dims = (N, C, H, W, K, R, S, ph, pw, sh, sw, P, Q)
    return _call("conv2d_fwd", dims, _dtype_code(x), x, w, out, workspace, OP_FWD, stream, bias, beta, flip,
                 (dh, dw), groups)


def conv2d_fwd_noalloc(x, w, pad=0, stride=1, out=None, stream=None):
    """Forward with no workspace: the library stages the repacked filter in its own fixed
    8 MiB device scratch, for callers that cannot allocate device memory.  Raises
    Conv2dError (CONV2D_ERR_NOALLOC_LIMIT) if the filter does not fit.  Calls that overlap
    on the GPU race on the shared scratch; keep them ordered on one stream."""
    import torch
    _check_tensor(x, "x")
    _check_tensor(w, "w")
    N, C, H, W = x.shape
    K, C2, R, S = w.shape
    if C2 != C or w.dtype != x.dtype:
        raise ValueError("x / w channel count or dtype mismatch")
    ph, pw = _pair(pad)
    sh, sw = _pair(stride)
    P, Q = conv2d_output_dim(H, ph, R, sh), conv2d_output_dim(W, pw, S, sw)
    if out is None:
        out = torch.empty((N, K, P, Q), dtype=x.dtype, device=x.device)
    rc = load_library().conv2d_fwd_noalloc(N, C, H, W, K, R, S, ph, pw, sh, sw, P, Q, _dtype_code(x),
                                           ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                           ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream))
    if rc:
        raise Conv2dError(rc, "conv2d_fwd_noalloc")
    return out


def conv2d_bwd_data(dy, w, x_hw, pad=0, stride=1, out=None, workspace=None, stream=None, bias=None, beta=0.0,
                    flip=False, dilation=1, groups=1):
    """dx (N,C,H,W) from dy (N,K,P,Q) and w (K,C,R,S); x_hw = (H, W).  Optional epilogue:
    + bias[c] (the bias of a deconvolution) + beta * dx (`out` required when beta != 0)."""
    import torch
    _check_tensor(dy, "dy")
    _check_tensor(w, "w")
    N, K, P, Q = dy.shape
    K2, Cg, R, S = w.shape
    C = Cg * groups
    if K2 != K or K % groups != 0 or w.dtype != dy.dtype:
        raise ValueError("dy / w channel count, groups or dtype mismatch")
    H, W = x_hw
    ph, pw = _pair(pad)
    sh, sw = _pair(stride)
    if out is None:
        if beta != 0.0:
            raise ValueError("beta != 0 accumulates onto `out`, which must then be given")
        out = torch.empty((N, C, H, W), dtype=dy.dtype, device=dy.device)
    _check_vec(bias, C, dy, "bias")
    dims = (N, C, H, W, K, R, S, ph, pw, sh, sw, P, Q)
    return _call("conv2d_bwd_data", dims, _dtype_code(dy), dy, w, out, workspace, OP_BWD_DATA, stream,
                 bias, beta, flip, _pair(dilation), groups)


def conv2d_bwd_filter(x, dy, rs, pad=0, stride=1, out=None, workspace=None, stream=None, beta=0.0,
                      db_k=None, db_c=None, flip=False, dilation=1, groups=1):
    """dw (K,C,R,S) from x (N,C,H,W) and dy (N,K,P,Q); rs = (R, S).

    Optional: beta accumulates onto `out` (dw) and onto the bias gradients; db_k (K values)
    receives sum of dy over (n, p, q) -- the convolution bias gradient; db_c (C values)
    receives sum of x over (n, h, w) -- the deconvolution bias gradient, x being the
    deconvolution's output gradient."""
    import torch
    _check_tensor(x, "x")
    _check_tensor(dy, "dy")
    N, C, H, W = x.shape
    N2, K, P, Q = dy.shape
    if N2 != N or dy.dtype != x.dtype:
        raise ValueError("x / dy batch or dtype mismatch")
    R, S = rs
    ph, pw = _pair(pad)
    sh, sw = _pair(stride)
    if out is None:
        if beta != 0.0:
            raise ValueError("beta != 0 accumulates onto `out`, which must then be given")
        out = torch.empty((K, C // groups, R, S), dtype=x.dtype, device=x.device)
    if C % groups != 0 or K % groups != 0:
        raise ValueError("groups must divide C and K")
    _check_vec(db_k, K, x, "db_k")
    _check_vec(db_c, C, x, "db_c")
    dims = (N, C, H, W, K, R, S, ph, pw, sh, sw, P, Q)
    dt = _dtype_code(x)
    dh, dw = _pair(dilation)
    ws, wsb = _workspace(OP_BWD_FILTER, dims, dt, workspace, out.device, (dh, dw), groups)
    rc = load_library().conv2d_bwd_filter_ex(*[int(v) for v in dims], dh, dw, int(groups), dt, _mode(flip), _ptr(x),
                                             _ptr(dy),
                                             ctypes.c_float(float(beta)), _ptr(out), _ptr(db_k), _ptr(db_c),
                                             _ptr(ws), ctypes.c_size_t(wsb), _stream_ptr(stream))
    if rc:
        raise Conv2dError(rc, "conv2d_bwd_filter")
    return out


def deconv2d_fwd(inp, wt, out_hw, pad=0, stride=1, out=None, workspace=None, stream=None, bias=None, beta=0.0,
                 flip=False, dilation=1, groups=1):
    """Transposed convolution: inp (N,Ci,Hi,Wi), wt (Ci,Co,R,S) -> (N,Co,Ho,Wo), optionally
    + bias[co] + beta * out.

    Runs conv2d_bwd_data with K = Ci (deconv input channels), C = Co, P = Hi, H = Ho."""
    return conv2d_bwd_data(inp, wt, out_hw, pad, stride, out=out, workspace=workspace, stream=stream,
                           bias=bias, beta=beta, flip=flip, dilation=dilation, groups=groups)


# ------------------------------------------------------------------ 1-D
# A 1-D convolution over (N, C, W) is the 2-D one with H = R = 1 (pad and stride along W
# only); these wrappers only reshape views and call the 2-D entry points.

def _one(v):
    return int(v if isinstance(v, int) else v[0])


def conv1d_fwd(x, w, pad=0, stride=1, out=None, workspace=None, stream=None, bias=None, beta=0.0, flip=False,
               dilation=1):
    """y (N,K,Q) = conv1d(x (N,C,W), w (K,C,S))."""
    o4 = out.unsqueeze(2) if out is not None else None
    y = conv2d_fwd(x.unsqueeze(2), w.unsqueeze(2), (0, _one(pad)), (1, _one(stride)), out=o4,
                   workspace=workspace, stream=stream, bias=bias, beta=beta, flip=flip, dilation=(1, _one(dilation)))
    return y.squeeze(2) if out is None else out


def conv1d_bwd_data(dy, w, x_w, pad=0, stride=1, out=None, workspace=None, stream=None, bias=None, beta=0.0,
                    flip=False, dilation=1):
    """dx (N,C,W) from dy (N,K,Q) and w (K,C,S); x_w = W."""
    o4 = out.unsqueeze(2) if out is not None else None
    dx = conv2d_bwd_data(dy.unsqueeze(2), w.unsqueeze(2), (1, int(x_w)), (0, _one(pad)), (1, _one(stride)), out=o4,
                         workspace=workspace, stream=stream, bias=bias, beta=beta, flip=flip,
                         dilation=(1, _one(dilation)))
    return dx.squeeze(2) if out is None else out


def conv1d_bwd_filter(x, dy, s, pad=0, stride=1, out=None, workspace=None, stream=None, beta=0.0, db_k=None,
                      db_c=None, flip=False, dilation=1):
    """dw (K,C,S) from x (N,C,W) and dy (N,K,Q); s = S."""
    o4 = out.unsqueeze(2) if out is not None else None
    dw = conv2d_bwd_filter(x.unsqueeze(2), dy.unsqueeze(2), (1, int(s)), (0, _one(pad)), (1, _one(stride)), out=o4,
                           workspace=workspace, stream=stream, beta=beta, db_k=db_k, db_c=db_c, flip=flip,
                           dilation=(1, _one(dilation)))
    return dw.squeeze(2) if out is None else out


def conv2d_kernel_launches() -> int:
    """Kernels the library has enqueued in this process so far (diagnostic counter)."""
    return int(load_library().conv2d_kernel_launches())


def conv2d_device_status(stream=None) -> int:
    """Synchronize the stream; raise if a kernel's bounded wait expired or the stream failed."""
    rc = load_library().conv2d_device_status(_stream_ptr(stream))
    if rc:
        raise Conv2dError(rc, "conv2d_device_status")
    return 0


def conv2d_bwd(x, w, dy, pad=0, stride=1, dx=None, dw=None, workspace=None, stream=None):
    """(dx, dw) = (conv2d_bwd_data(dy, w), conv2d_bwd_filter(x, dy)) in one call; with bf16
    tensors dy is read from memory once for both where the plans allow."""
    import torch
    for t, nm in ((x, "x"), (w, "w"), (dy, "dy")):
        _check_tensor(t, nm)
    N, C, H, W = x.shape
    K, C2, R, S = w.shape
    if C2 != C or w.dtype != x.dtype or dy.dtype != x.dtype:
        raise ValueError("x / w channel count or dtype mismatch")
    ph, pw = _pair(pad)
    sh, sw = _pair(stride)
    P, Q = conv2d_output_dim(H, ph, R, sh), conv2d_output_dim(W, pw, S, sw)
    if tuple(dy.shape) != (N, K, P, Q):
        raise ValueError("dy shape does not match the descriptor")
    dims = (N, C, H, W, K, R, S, ph, pw, sh, sw, P, Q)
    dt = _dtype_code(x)
    if dx is None:
        dx = torch.empty_like(x)
    if dw is None:
        dw = torch.empty_like(w)
    ws, wsb = _workspace(OP_BWD, dims, dt, workspace, x.device)
    rc = load_library().conv2d_bwd(*dims, dt, _ptr(x), _ptr(w), _ptr(dy), _ptr(dx), _ptr(dw), _ptr(ws),
                                   ctypes.c_size_t(wsb), _stream_ptr(stream))
    if rc:
        raise Conv2dError(rc, "conv2d_bwd")
    return dx, dw


# ---------------------------------------------------------------------------- 3-D (NCDHW)
def _triple(v):
    return (int(v),) * 3 if isinstance(v, int) else tuple(int(a) for a in v)


def _dims3(N, C, dhw, K, trs, pad, stride, dilation):
    pads, strides, dils = _triple(pad), _triple(stride), _triple(dilation)
    out = [conv2d_output_dim(i_, p_, d_ * (k_ - 1) + 1, s_) for i_, p_, k_, s_, d_ in zip(dhw, pads, trs, strides, dils)]
    return [N, C, *dhw, K, *trs, *pads, *strides, *dils, *out], tuple(out)


def _call3(name, dims, groups, dt, a, b, out, workspace, op, stream):
    import torch
    arr = (ctypes.c_int * 21)(*dims)
    need = ctypes.c_size_t(0)
    rc = load_library().conv3d_workspace_size(op, arr, int(groups), dt, ctypes.byref(need))
    if rc:
        raise Conv2dError(rc, "conv3d_workspace_size")
    if workspace is None:
        workspace = torch.empty(max(need.value, 1), dtype=torch.uint8, device=out.device)
    if workspace.numel() * workspace.element_size() < need.value:
        raise ValueError(f"workspace too small: need {need.value} bytes")
    rc = getattr(load_library(), name)(arr, int(groups), dt, _ptr(a), _ptr(b), _ptr(out), _ptr(workspace),
                                       ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                                       _stream_ptr(stream))
    if rc:
        raise Conv2dError(rc, name)
    return out


def conv3d_fwd(x, w, pad=0, stride=1, dilation=1, groups=1, out=None, workspace=None, stream=None):
    """y (N,K,Z,P,Q) = 3-D cross-correlation of x (N,C,D,H,W) with w (K,C/groups,T,R,S)."""
    import torch
    _check_tensor(x, "x")
    _check_tensor(w, "w")
    N, C = x.shape[:2]
    K, Cg = w.shape[:2]
    if Cg * groups != C or K % groups != 0 or w.dtype != x.dtype:
        raise ValueError("x / w channel count, groups or dtype mismatch")
    dims, zpq = _dims3(N, C, tuple(x.shape[2:]), K, tuple(w.shape[2:]), pad, stride, dilation)
    if out is None:
        out = torch.empty((N, K, *zpq), dtype=x.dtype, device=x.device)
    return _call3("conv3d_fwd", dims, groups, _dtype_code(x), x, w, out, workspace, OP_FWD, stream)


def conv3d_bwd_data(dy, w, x_dhw, pad=0, stride=1, dilation=1, groups=1, out=None, workspace=None, stream=None):
    """dx (N,C,D,H,W) from dy (N,K,Z,P,Q) and w (K,C/groups,T,R,S); x_dhw = (D, H, W)."""
    import torch
    _check_tensor(dy, "dy")
    _check_tensor(w, "w")
    N, K = dy.shape[:2]
    K2, Cg = w.shape[:2]
    if K2 != K or K % groups != 0 or w.dtype != dy.dtype:
        raise ValueError("dy / w channel count, groups or dtype mismatch")
    C = Cg * groups
    dims, zpq = _dims3(N, C, tuple(x_dhw), K, tuple(w.shape[2:]), pad, stride, dilation)
    if tuple(dy.shape[2:]) != zpq:
        raise ValueError("dy spatial shape does not match the descriptor")
    if out is None:
        out = torch.empty((N, C, *x_dhw), dtype=dy.dtype, device=dy.device)
    return _call3("conv3d_bwd_data", dims, groups, _dtype_code(dy), dy, w, out, workspace, OP_BWD_DATA, stream)


def conv3d_bwd_filter(x, dy, trs, pad=0, stride=1, dilation=1, groups=1, out=None, workspace=None, stream=None):
    """dw (K,C/groups,T,R,S) from x (N,C,D,H,W) and dy (N,K,Z,P,Q); trs = (T, R, S)."""
    import torch
    _check_tensor(x, "x")
    _check_tensor(dy, "dy")
    N, C = x.shape[:2]
    K = dy.shape[1]
    if C % groups != 0 or K % groups != 0 or dy.dtype != x.dtype:
        raise ValueError("x / dy channel count, groups or dtype mismatch")
    dims, zpq = _dims3(N, C, tuple(x.shape[2:]), K, tuple(trs), pad, stride, dilation)
    if tuple(dy.shape[2:]) != zpq:
        raise ValueError("dy spatial shape does not match the descriptor")
    if out is None:
        out = torch.empty((K, C // groups, *trs), dtype=x.dtype, device=x.device)
    return _call3("conv3d_bwd_filter", dims, groups, _dtype_code(x), x, dy, out, workspace, OP_BWD_FILTER, stream)

/*
 * conv2d_gb300.h -- C ABI of the GB300 (sm_103a) NCHW 2-D convolution library.
 *
 * Three operations of dense 2-D cross-correlation with zero padding and stride,
 * described by the thirteen integers N, C, H, W, K, R, S, pad_h, pad_w, stride_h,
 * stride_w, P, Q in the order of the cuDNN wrapper factory methods of Apache
 * SystemDS (page "LibMatrixCuDNNConvolutionAlgorithm.java",
 * cudnnGetConvolutionForwardAlgorithm / ...BackwardFilterAlgorithm /
 * ...BackwardDataAlgorithm parameter lists):
 *
 *   x  : N x C x H x W   (NCHW, dense, row-major)        "nchwTensorDesc"
 *   w  : K x C x R x S   (KCRS, dense, row-major)        "filterDesc"
 *   y  : N x K x P x Q   (dense, row-major)              "nkpqTensorDesc"
 *   P  = floor((H + 2*pad_h - R) / stride_h) + 1,  Q likewise with W, pad_w, S, stride_w
 *   X(n,c,h,w) = x[n,c,h,w] inside the image, 0 outside (zero padding)
 *
 *   forward          y[n,k,p,q]  = sum_{c,r,s} X(n,c,p*stride_h-pad_h+r,q*stride_w-pad_w+s) * w[k,c,r,s]
 *   backward-data    dx[n,c,h,w] = sum over (k,r,s,p,q) with h = p*stride_h-pad_h+r and
 *                                  w = q*stride_w-pad_w+s of dy[n,k,p,q] * w[k,c,r,s]
 *   backward-filter  dw[k,c,r,s] = sum_{n,p,q} X(n,c,p*stride_h-pad_h+r,q*stride_w-pad_w+s) * dy[n,k,p,q]
 *
 * The mode is cross-correlation with dilation 1 (same page,
 * allocateConvolutionDescriptor: CUDNN_CROSS_CORRELATION, dilation 1,1).  Outputs
 * are overwritten, never accumulated: alpha = 1, beta = 0 as in the ConvolutionForward
 * / ConvolutionBackwardData / ConvolutionBackwardFilter calls of the C# examples page
 * ("FilterDescriptor.SetFilter4dDescriptor" examples: Conv2D, DoConvolutionGradient).
 *
 * Transposed convolution (deconvolution) forward is conv2d_bwd_data with the weight
 * read as (deconv_in, deconv_out, R, S) = (K, C, R, S): deconv input = dy (N,K,P,Q),
 * deconv output = dx (N,C,H,W).  Its backward-data is conv2d_fwd and its
 * backward-weights is conv2d_bwd_filter with x = deconv output gradient and
 * dy = deconv input (page "mkldnn_deconvolution.cc", MKLDNNDeconvFwd::Execute comment).
 * H and W are explicit arguments because for stride > 1 several H give the same P.
 *
 * Data types (page "mkldnn_deconvolution.cc", SupportMKLDNNDeconv: float32 or bfloat16):
 *   CONV2D_DTYPE_F32   fp32 tensors; products on TF32 tensor cores, fp32 accumulation.
 *   CONV2D_DTYPE_BF16  bf16 tensors; bf16 products, fp32 accumulation, bf16 output
 *                      rounded to nearest even.
 *
 * Memory, streams, ownership:
 *   - All tensor pointers are DEVICE pointers owned by the caller, aligned to the
 *     element size.  Inputs are read-only.  Outputs must not alias inputs.
 *   - `workspace` is caller-owned device memory of at least the size reported by
 *     conv2d_workspace_size() for the same op and descriptor, 16-byte aligned.  The
 *     size never exceeds 1e9 bytes (the workspace cap of the SystemDS wrapper,
 *     MAX_WORKSPACE_LIMIT_BYTES).  Forward and backward-data stage a repacked copy of
 *     the filter there; backward-filter stages split partial sums, and with a stride
 *     above 1 (dilation 1) also a copy of x rearranged into its stride phases.
 *   - Forward and backward-data with large filters over many source channels (about
 *     13 x 13 taps and more) run as several passes over contiguous ranges of the taps
 *     r*S + s, each adding onto the output the previous one wrote; with bf16 tensors
 *     the output is then rounded to bf16 once per pass.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only enqueue
 *     work on it and return; the library allocates no device memory, keeps no
 *     pointer after returning and holds no per-call state.  Results are
 *     deterministic run to run.
 *
 * Errors: every function returns CONV2D_OK (0) or a negative code; nothing throws or
 * aborts.  Argument errors are detected on the host before anything is enqueued.
 * A kernel whose internal pipeline wait exceeds its time limit (about one second)
 * stops early and records CONV2D_ERR_DEVICE_TIMEOUT, which conv2d_device_status()
 * reports.
 */
#ifndef CONV2D_GB300_H
#define CONV2D_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    CONV2D_DTYPE_F32 = 0,
    CONV2D_DTYPE_BF16 = 1
};

/* Convolution mode (cuDNN's cudnnConvolutionMode_t, which the SystemDS page sets to
 * CUDNN_CROSS_CORRELATION in allocateConvolutionDescriptor): cross-correlation (the
 * formulas above), or convolution, the same with the filter rotated by 180 degrees --
 * tap (r, s) multiplies w[k,c,R-1-r,S-1-s]; its backward-filter returns the gradient of that
 * filter, dw[k,c,R-1-r,S-1-s] = the cross-correlation dw[k,c,r,s].  Only the _ex entry points
 * take a mode; the plain ones are cross-correlation. */
enum {
    CONV2D_MODE_CROSS_CORRELATION = 0,
    CONV2D_MODE_CONVOLUTION = 1
};

enum {
    CONV2D_OP_FWD = 0,
    CONV2D_OP_BWD_DATA = 1,
    CONV2D_OP_BWD_FILTER = 2,
    CONV2D_OP_BWD = 3           /* both gradients in one call (conv2d_bwd) */
};

enum {
    CONV2D_OK = 0,
    CONV2D_ERR_BAD_DESC = -1,       /* a dimension <= 0, pad < 0 or stride < 1 */
    CONV2D_ERR_SHAPE = -2,          /* P or Q differs from the formula, or is < 1 */
    CONV2D_ERR_NULLPTR = -3,        /* a tensor pointer (or a needed workspace) is NULL */
    CONV2D_ERR_ALIGN = -4,          /* a pointer is not aligned as documented above */
    CONV2D_ERR_DTYPE = -5,          /* unknown dtype */
    CONV2D_ERR_WORKSPACE = -6,      /* workspace_bytes below conv2d_workspace_size() */
    CONV2D_ERR_TOO_LARGE = -7,      /* a tensor has >= 2^31 elements */
    CONV2D_ERR_LAUNCH = -8,         /* the CUDA runtime rejected a launch */
    CONV2D_ERR_DEVICE = -9,         /* no usable sm_100-family device */
    CONV2D_ERR_DEVICE_TIMEOUT = -10,/* a kernel's bounded internal wait expired */
    CONV2D_ERR_UNSUPPORTED = -11,   /* R*S > 4096, stride_h*stride_w > 64, or no tile fits
                                       shared memory: forward / backward-data even with the
                                       taps split over 16 passes of at most 256 taps,
                                       backward-filter with more than 256 taps in one stride
                                       phase or when the dilated filter spans too many input
                                       rows */
    CONV2D_ERR_BAD_OP = -12,        /* unknown op in conv2d_workspace_size() */
    CONV2D_ERR_NOALLOC_LIMIT = -13  /* conv2d_fwd_noalloc: problem exceeds its fixed scratch */
};

/* Output extent of one spatial dimension: *out = floor((in + 2*pad - k)/stride) + 1.
 * Returns CONV2D_ERR_BAD_DESC for in, k <= 0, pad < 0, stride < 1 or a NULL out, and
 * CONV2D_ERR_SHAPE when the padded input is shorter than the filter. */
int conv2d_output_dim(int in, int pad, int k, int stride, int *out);

/* Bytes of device workspace `op` needs for this descriptor and dtype (<= 1e9).
 * Validates the descriptor exactly as the op itself does. */
int conv2d_workspace_size(int op, int N, int C, int H, int W, int K, int R, int S,
                          int pad_h, int pad_w, int stride_h, int stride_w, int P, int Q,
                          int dtype, size_t *bytes);

/* conv2d_workspace_size for a dilated and/or grouped descriptor (dil_h = dil_w = groups = 1:
 * the same value). */
int conv2d_workspace_size_ex(int op, int N, int C, int H, int W, int K, int R, int S,
                             int pad_h, int pad_w, int stride_h, int stride_w, int P, int Q,
                             int dil_h, int dil_w, int groups, int dtype, size_t *bytes);

/* Forward: y (N,K,P,Q) = conv(x (N,C,H,W), w (K,C,R,S)). */
int conv2d_fwd(int N, int C, int H, int W, int K, int R, int S,
               int pad_h, int pad_w, int stride_h, int stride_w, int P, int Q, int dtype,
               const void *x, const void *w, void *y,
               void *workspace, size_t workspace_bytes, void *stream);

/* Backward-data (= deconvolution forward): dx (N,C,H,W) from dy (N,K,P,Q) and w (K,C,R,S).
 * Every element of dx is written; elements no output window reads are 0. */
int conv2d_bwd_data(int N, int C, int H, int W, int K, int R, int S,
                    int pad_h, int pad_w, int stride_h, int stride_w, int P, int Q, int dtype,
                    const void *dy, const void *w, void *dx,
                    void *workspace, size_t workspace_bytes, void *stream);

/* Backward-filter: dw (K,C,R,S) from x (N,C,H,W) and dy (N,K,P,Q). */
int conv2d_bwd_filter(int N, int C, int H, int W, int K, int R, int S,
                      int pad_h, int pad_w, int stride_h, int stride_w, int P, int Q, int dtype,
                      const void *x, const void *dy, void *dw,
                      void *workspace, size_t workspace_bytes, void *stream);

/* Fused epilogues (page "mkldnn_deconvolution.cc": the deconvolution forward takes an
 * optional bias and an output request that either writes or adds to the output
 * (MKLDNNDeconvFwd::Execute, OutMem(req, ...)); its backward-weights pass also produces
 * the bias gradient (ScheduleBwdWeights: bias_req, BiasGradMem).  cuDNN's alpha/beta
 * scaling of the C# examples page is the same output rule with alpha = 1.)
 *
 * Each result element is computed in fp32 as  D + bias[channel] + beta * old  and then
 * stored (bf16: rounded to nearest even), where D is the op's sum above, `old` the value
 * the output held before the call (read only when beta != 0), and the bias term applies
 * only where a bias pointer is given.  beta = 0 overwrites (the plain entry points);
 * beta = 1 accumulates (MXNet kAddTo).  bias / db vectors have the tensor dtype, are
 * device pointers aligned to the element size, and must not alias any other argument.
 *
 * conv2d_fwd_ex:       y = conv(x, w) + bias[k] + beta * y;            bias: K values or NULL.
 * conv2d_bwd_data_ex:  dx = bwd_data(dy, w) + bias[c] + beta * dx;      bias: C values or NULL
 *                      (the bias of a deconvolution, whose output is dx).
 * conv2d_bwd_filter_ex: dw = bwd_filter(x, dy) + beta * dw, and optionally
 *                      db_k[k] = sum_{n,p,q} dy[n,k,p,q] + beta * db_k[k]  (convolution bias
 *                                gradient; K values), and
 *                      db_c[c] = sum_{n,h,w} x[n,c,h,w] + beta * db_c[c]   (deconvolution bias
 *                                gradient: x is the deconvolution's output gradient; C values).
 *                      Either may be NULL.  Sums are in fixed order (deterministic).  When a
 *                      bias gradient is requested the workspace must have the full size
 *                      conv2d_workspace_size(CONV2D_OP_BWD_FILTER, ...) reports; otherwise the
 *                      split partials alone suffice.
 * `mode` is CONV2D_MODE_CROSS_CORRELATION or CONV2D_MODE_CONVOLUTION (any other value:
 * CONV2D_ERR_BAD_DESC).  dil_h, dil_w >= 1 are the filter dilation (cuDNN's dilation of the
 * convolution descriptor, which the SystemDS page sets to 1, 1): filter tap (r, s) reads
 * X(n, c, p*stride_h - pad_h + r*dil_h, q*stride_w - pad_w + s*dil_w), and
 * P = floor((H + 2*pad_h - dil_h*(R-1) - 1) / stride_h) + 1, Q likewise; the workspace of a
 * dilated problem is sized by conv2d_workspace_size_ex.  groups >= 1 divides C and K: the
 * channels split into `groups` independent convolutions (input channels g*C/groups .. and output
 * channels g*K/groups .. of group g), and the filter is K x C/groups x R x S (cuDNN's
 * group count of the convolution descriptor); C and K stay the tensors' channel counts.  Same descriptors, workspace rules and error codes as the plain
 * entry points (which are these with cross-correlation, bias = NULL, beta = 0,
 * db_k = db_c = NULL). */
int conv2d_fwd_ex(int N, int C, int H, int W, int K, int R, int S,
                  int pad_h, int pad_w, int stride_h, int stride_w, int P, int Q,
                  int dil_h, int dil_w, int groups, int dtype, int mode,
                  const void *x, const void *w, const void *bias, float beta, void *y,
                  void *workspace, size_t workspace_bytes, void *stream);

int conv2d_bwd_data_ex(int N, int C, int H, int W, int K, int R, int S,
                       int pad_h, int pad_w, int stride_h, int stride_w, int P, int Q,
                       int dil_h, int dil_w, int groups, int dtype, int mode,
                       const void *dy, const void *w, const void *bias, float beta, void *dx,
                       void *workspace, size_t workspace_bytes, void *stream);

int conv2d_bwd_filter_ex(int N, int C, int H, int W, int K, int R, int S,
                         int pad_h, int pad_w, int stride_h, int stride_w, int P, int Q,
                         int dil_h, int dil_w, int groups, int dtype, int mode,
                         const void *x, const void *dy, float beta, void *dw, void *db_k, void *db_c,
                         void *workspace, size_t workspace_bytes, void *stream);

/* Both gradients of one convolution in one call: dx = conv2d_bwd_data(dy, w) and
 * dw = conv2d_bwd_filter(x, dy), overwritten, cross-correlation (page "mkldnn_deconvolution.cc",
 * MKLDNNDeconvBwd::Execute: backward-data and backward-weights scheduled together on the shared
 * output gradient).  With bf16 tensors, where the backward-data plan stages dy from the same
 * channel-chunk copy that the backward-filter plan makes, dy is read from memory once for both;
 * otherwise the two operations run one after the other.  Same descriptor, pointer and error
 * rules as the single operations; the workspace is sized by conv2d_workspace_size with
 * CONV2D_OP_BWD. */
int conv2d_bwd(int N, int C, int H, int W, int K, int R, int S,
               int pad_h, int pad_w, int stride_h, int stride_w, int P, int Q,
               int dtype, const void *x, const void *w, const void *dy, void *dx, void *dw,
               void *workspace, size_t workspace_bytes, void *stream);

/* 3-D (NCDHW) cross-correlation, the same three operations one dimension up (page
 * "mkldnn_deconvolution.cc": SupportMKLDNNDeconv accepts kernels of 1 to 3 spatial dimensions,
 * DeconvDescCreator strides, pads and dilations of the same rank):
 *
 *   x  : N x C x D x H x W,  w : K x C/groups x T x R x S,  y : N x K x Z x P x Q
 *   y[n,k,z,p,q] = sum_{c,t,r,s} X(n, c, z*stride_d - pad_d + t*dil_d,
 *                                        p*stride_h - pad_h + r*dil_h, q*stride_w - pad_w + s*dil_w) * w[k,c,t,r,s]
 *   (X zero outside the tensor; c over the input channels of k's group); backward-data and
 *   backward-filter are its two gradients, as in 2-D.
 *
 * `dims` points to 21 host ints: N, C, D, H, W, K, T, R, S, pad_d, pad_h, pad_w, stride_d,
 * stride_h, stride_w, dil_d, dil_h, dil_w, Z, P, Q (Z, P, Q by the dilated floor formula, else
 * CONV2D_ERR_SHAPE).  groups >= 1 divides C and K.  Outputs are overwritten (beta = 0),
 * cross-correlation.  Each op runs as one 2-D operation per depth tap t on a batch of the N*Z
 * depth slices that tap reads (gathered into the workspace), so the 2-D limits apply to
 * (R, S, strides, dilations) and the workspace (256-byte aligned) must hold
 * conv3d_workspace_size() bytes: the gathered batches, one filter slice, for backward-data an
 * fp32 dx accumulator, and the 2-D call's workspace.  bf16 forward outputs are rounded once per
 * depth tap (the passes add onto the output); backward-data accumulates in fp32. */
int conv3d_workspace_size(int op, const int *dims, int groups, int dtype, size_t *bytes);
int conv3d_fwd(const int *dims, int groups, int dtype, const void *x, const void *w, void *y,
               void *workspace, size_t workspace_bytes, void *stream);
int conv3d_bwd_data(const int *dims, int groups, int dtype, const void *dy, const void *w, void *dx,
                    void *workspace, size_t workspace_bytes, void *stream);
int conv3d_bwd_filter(const int *dims, int groups, int dtype, const void *x, const void *dy, void *dw,
                      void *workspace, size_t workspace_bytes, void *stream);

/* Forward without any workspace argument, for callers that cannot allocate device
 * memory: for example code whose device memory is entirely owned by another runtime's
 * pool, or a latency-critical path that must never call cudaMalloc (which can
 * synchronize the device).  There is no counterpart of this entry point on the
 * reference pages; it is an addition of this library.
 *
 * Same arguments, layouts, results and error codes as conv2d_fwd (the same plan, large
 * filters included: their tap passes each stage a repacked filter slice), except that the
 * repacked filter is staged in a fixed 8 MiB scratch array compiled into the library
 * instead of a caller workspace.  The function itself allocates nothing.
 *   - Limit: returns CONV2D_ERR_NOALLOC_LIMIT (nothing enqueued) when the repacked
 *     filter needs more than 8 MiB, which is about 2M fp32 or 4M bf16 filter values
 *     (rounded up to whole tiles); conv2d_workspace_size(CONV2D_OP_FWD, ...) reports the
 *     size needed, and every size up to and including 8 MiB is accepted.
 *   - The scratch exists once per GPU that loaded the library and is held until the
 *     process exits.  The first call on a device looks up the scratch's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call before
 *     any stream capture.
 *   - All calls share the scratch and it keeps the last call's contents (each call
 *     rewrites the part it uses before reading it).  Calls whose execution overlaps on
 *     the GPU (different streams, no ordering) race on it: order them on one stream or
 *     with events. */
int conv2d_fwd_noalloc(int N, int C, int H, int W, int K, int R, int S,
                       int pad_h, int pad_w, int stride_h, int stride_w, int P, int Q, int dtype,
                       const void *x, const void *w, void *y, void *stream);

/* Synchronizes `stream`, then reports CONV2D_ERR_DEVICE_TIMEOUT if any kernel of this
 * library hit its bounded-wait limit since the previous call (and clears the record),
 * CONV2D_ERR_LAUNCH if the stream reports a CUDA error, else CONV2D_OK. */
int conv2d_device_status(void *stream);

/* Number of kernels the library has enqueued in this process so far, on any stream and
 * device (a diagnostic: the difference across a region counts the kernels the region's
 * calls launched).  Thread-safe. */
unsigned long long conv2d_kernel_launches(void);

/* Static description of an error code. */
const char *conv2d_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* CONV2D_GB300_H */

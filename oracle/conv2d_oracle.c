/*
 * conv2d_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct fp64 CPU implementation of dense NCHW 2-D
 * cross-correlation with zero padding and stride, and of its two gradients.
 * It exists to check the CUDA path; the product never links or calls it.
 * Only the tests, the smoke check and the CPU-baseline leg of the bench may
 * load this file's shared library.
 *
 * Notation (Apache SystemDS, LibMatrixCuDNNConvolutionAlgorithm.java, the
 * factory-method parameter lists): N images, C channels, H x W image, K output
 * "channels", R x S filter, pad_h/pad_w, stride_h/stride_w, P x Q output.
 * Layouts (same page, allocateTensorDescriptor / allocateFilterDescriptor):
 * x is NCHW, y and dy are N,K,P,Q, the filter w is K,C,R,S.  The mode is
 * CUDNN_CROSS_CORRELATION with dilation 1,1 (allocateConvolutionDescriptor).
 * Outputs are overwritten (alpha = 1, beta = 0, as in the C# Conv2D /
 * DoConvolutionGradient examples of the third page).
 *
 * Every result below is the literal definition, summed in fp64, one output
 * element at a time (gather form).  No blocking, no reordering beyond the
 * order the definition is written in.  OpenMP splits the outer loops over
 * output elements; each output is owned by one thread, so the result is
 * deterministic.
 *
 * Parity status: every function here is pinned by the CPU tests
 * (tests/test_oracle_pins.py): P/Q by window enumeration, 1x1 = matmul,
 * delta filter = shifted copy, the adjoint identity across the three ops,
 * the dense-operator transpose, the scatter-form deconvolution, hand-counted
 * golden values, and an independent library witness.  NaN/Inf propagation is
 * parity unpinned (inputs are finite everywhere).
 */
#include <stddef.h>
#include <stdint.h>

#define IDX4(a, b, c, d, B, C, D) ((((int64_t)(a) * (B) + (b)) * (C) + (c)) * (D) + (d))

/* Output extent of one spatial dimension: the number of window positions
 * p >= 0 with p*stride - pad + (k-1) <= in - 1 + pad, i.e.
 * floor((in + 2*pad - k)/stride) + 1, or 0 when the padded input is shorter
 * than the filter.  The pages pass P and Q in; this is the plain reading of
 * how they relate to H, pad_h, R and stride_h. */
int oracle_output_dim(int in, int pad, int k, int stride)
{
    if (in <= 0 || pad < 0 || k <= 0 || stride <= 0)
        return -1;
    int num = in + 2 * pad - k;
    if (num < 0)
        return 0;
    return num / stride + 1;
}

/* Zero-padded read of x[n,c,h,w]. */
static inline double xpad(const double *x, int n, int c, int h, int w, int C, int H, int W)
{
    if (h < 0 || h >= H || w < 0 || w >= W)
        return 0.0;
    return x[IDX4(n, c, h, w, C, H, W)];
}

/* Forward: y[n,k,p,q] = sum_{c,r,s} X(n,c,p*sh-ph+r,q*sw-pw+s) * w[k,c,r,s]. */
static double fwd_one(const double *x, const double *w, int n, int k, int p, int q,
                      int C, int H, int W, int R, int S, int ph, int pw, int sh, int sw)
{
    double acc = 0.0;
    for (int c = 0; c < C; ++c)
        for (int r = 0; r < R; ++r)
            for (int s = 0; s < S; ++s)
                acc += xpad(x, n, c, p * sh - ph + r, q * sw - pw + s, C, H, W) *
                       w[IDX4(k, c, r, s, C, R, S)];
    return acc;
}

void oracle_conv2d_fwd(const double *x, const double *w, double *y,
                       int N, int C, int H, int W, int K, int R, int S,
                       int ph, int pw, int sh, int sw, int P, int Q)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            for (int p = 0; p < P; ++p)
                for (int q = 0; q < Q; ++q)
                    y[IDX4(n, k, p, q, K, P, Q)] =
                        fwd_one(x, w, n, k, p, q, C, H, W, R, S, ph, pw, sh, sw);
}

/* Backward data: dx[n,c,h,w] = sum over (k,r,s) of dy[n,k,p,q]*w[k,c,r,s]
 * where h = p*sh - ph + r and w = q*sw - pw + s for an output position
 * 0 <= p < P, 0 <= q < Q.  For a given (h, r) that position exists when
 * t = h + ph - r is >= 0, divisible by sh, and t/sh < P.  The sign test comes
 * before the divisibility test so that C's truncating % never sees a
 * negative operand.  Elements no output reads stay exactly 0. */
static double bwd_data_one(const double *dy, const double *w, int n, int c, int h, int ww,
                           int C, int K, int R, int S, int ph, int pw, int sh, int sw,
                           int P, int Q)
{
    double acc = 0.0;
    for (int k = 0; k < K; ++k)
        for (int r = 0; r < R; ++r) {
            int th = h + ph - r;
            if (th < 0 || th % sh != 0)
                continue;
            int p = th / sh;
            if (p >= P)
                continue;
            for (int s = 0; s < S; ++s) {
                int tw = ww + pw - s;
                if (tw < 0 || tw % sw != 0)
                    continue;
                int q = tw / sw;
                if (q >= Q)
                    continue;
                acc += dy[IDX4(n, k, p, q, K, P, Q)] * w[IDX4(k, c, r, s, C, R, S)];
            }
        }
    return acc;
}

void oracle_conv2d_bwd_data(const double *dy, const double *w, double *dx,
                            int N, int C, int H, int W, int K, int R, int S,
                            int ph, int pw, int sh, int sw, int P, int Q)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int n = 0; n < N; ++n)
        for (int c = 0; c < C; ++c)
            for (int h = 0; h < H; ++h)
                for (int ww = 0; ww < W; ++ww)
                    dx[IDX4(n, c, h, ww, C, H, W)] =
                        bwd_data_one(dy, w, n, c, h, ww, C, K, R, S, ph, pw, sh, sw, P, Q);
}

/* Backward filter: dw[k,c,r,s] = sum_{n,p,q} X(n,c,p*sh-ph+r,q*sw-pw+s) * dy[n,k,p,q]. */
static double bwd_filter_one(const double *x, const double *dy, int k, int c, int r, int s,
                             int N, int C, int H, int W, int K, int ph, int pw, int sh, int sw,
                             int P, int Q)
{
    double acc = 0.0;
    for (int n = 0; n < N; ++n)
        for (int p = 0; p < P; ++p)
            for (int q = 0; q < Q; ++q)
                acc += xpad(x, n, c, p * sh - ph + r, q * sw - pw + s, C, H, W) *
                       dy[IDX4(n, k, p, q, K, P, Q)];
    return acc;
}

void oracle_conv2d_bwd_filter(const double *x, const double *dy, double *dw,
                              int N, int C, int H, int W, int K, int R, int S,
                              int ph, int pw, int sh, int sw, int P, int Q)
{
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int k = 0; k < K; ++k)
        for (int c = 0; c < C; ++c)
            for (int r = 0; r < R; ++r)
                for (int s = 0; s < S; ++s)
                    dw[IDX4(k, c, r, s, C, R, S)] =
                        bwd_filter_one(x, dy, k, c, r, s, N, C, H, W, K, ph, pw, sh, sw, P, Q);
}

/* Transposed convolution ("deconvolution") forward, written in scatter form
 * straight from its own definition: every input element in[n,ci,p,q] adds
 * in*wt[ci,co,r,s] to out[n,co,p*sh-ph+r,q*sw-pw+s], targets outside the
 * output being dropped.  The weight is (deconv_in, deconv_out, R, S), the
 * "iohw" order of Apache MXNet's mkldnn_deconvolution.cc
 * (MKLDNNDeconvFwd::Execute comment).  This loop shares nothing with the
 * gather form above; the tests use it as an independent witness that
 * deconvolution forward equals convolution backward-data with K = deconv_in
 * and C = deconv_out.  Serial on purpose: scatter targets overlap. */
void oracle_deconv2d_fwd_scatter(const double *in, const double *wt, double *out,
                                 int N, int Ci, int Hi, int Wi, int Co, int R, int S,
                                 int ph, int pw, int sh, int sw, int Ho, int Wo)
{
    for (int64_t i = 0; i < (int64_t)N * Co * Ho * Wo; ++i)
        out[i] = 0.0;
    for (int n = 0; n < N; ++n)
        for (int ci = 0; ci < Ci; ++ci)
            for (int p = 0; p < Hi; ++p)
                for (int q = 0; q < Wi; ++q) {
                    double v = in[IDX4(n, ci, p, q, Ci, Hi, Wi)];
                    for (int co = 0; co < Co; ++co)
                        for (int r = 0; r < R; ++r) {
                            int oh = p * sh - ph + r;
                            if (oh < 0 || oh >= Ho)
                                continue;
                            for (int s = 0; s < S; ++s) {
                                int ow = q * sw - pw + s;
                                if (ow < 0 || ow >= Wo)
                                    continue;
                                out[IDX4(n, co, oh, ow, Co, Ho, Wo)] +=
                                    v * wt[IDX4(ci, co, r, s, Co, R, S)];
                            }
                        }
                }
}

/* Sampled evaluation: the same per-element definitions as above, evaluated
 * only at the flat output indices idx[0..count).  Used for parity at full
 * problem sizes, where computing every output on the CPU would take long. */
void oracle_conv2d_fwd_at(const double *x, const double *w,
                          int N, int C, int H, int W, int K, int R, int S,
                          int ph, int pw, int sh, int sw, int P, int Q,
                          const int64_t *idx, int64_t count, double *out)
{
    (void)N;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; ++i) {
        int64_t f = idx[i];
        int q = (int)(f % Q); f /= Q;
        int p = (int)(f % P); f /= P;
        int k = (int)(f % K); f /= K;
        int n = (int)f;
        out[i] = fwd_one(x, w, n, k, p, q, C, H, W, R, S, ph, pw, sh, sw);
    }
}

void oracle_conv2d_bwd_data_at(const double *dy, const double *w,
                               int N, int C, int H, int W, int K, int R, int S,
                               int ph, int pw, int sh, int sw, int P, int Q,
                               const int64_t *idx, int64_t count, double *out)
{
    (void)N;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; ++i) {
        int64_t f = idx[i];
        int ww = (int)(f % W); f /= W;
        int h = (int)(f % H); f /= H;
        int c = (int)(f % C); f /= C;
        int n = (int)f;
        out[i] = bwd_data_one(dy, w, n, c, h, ww, C, K, R, S, ph, pw, sh, sw, P, Q);
    }
}

void oracle_conv2d_bwd_filter_at(const double *x, const double *dy,
                                 int N, int C, int H, int W, int K, int R, int S,
                                 int ph, int pw, int sh, int sw, int P, int Q,
                                 const int64_t *idx, int64_t count, double *out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < count; ++i) {
        int64_t f = idx[i];
        int s = (int)(f % S); f /= S;
        int r = (int)(f % R); f /= R;
        int c = (int)(f % C); f /= C;
        int k = (int)f;
        out[i] = bwd_filter_one(x, dy, k, c, r, s, N, C, H, W, K, ph, pw, sh, sw, P, Q);
    }
}

/* Number of OpenMP threads a parallel region of this library uses. */
int oracle_num_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            extern int omp_get_num_threads(void);
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}

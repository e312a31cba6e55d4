/*
 * conv3d_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow fp64 CPU definitions of dense NCDHW 3-D cross-correlation with
 * zero padding, stride and dilation in each of the three spatial dims, and of
 * its two gradients.  Same role and rules as conv2d_oracle.c: the product
 * never links or calls it; only the tests, the smoke check and the bench's
 * CPU leg load this library.
 *
 * Source: Apache MXNet, mkldnn_deconvolution.cc -- SupportMKLDNNDeconv
 * accepts kernels of one to three spatial dims with an input
 * of two more dims (batch, channel), and the primitive setup takes one
 * stride, pad and dilation per spatial dim (CHECK_EQ of their counts, 1..3).
 * Notation extends the 2-D one by a depth dim in front: N images, C
 * channels, D x H x W input, K output channels, T x R x S filter, pads
 * pd/ph/pw, strides sd/sh/sw, dilations dd/dh/dw, Z x P x Q output.  Layouts:
 * x is N,C,D,H,W; y and dy are N,K,Z,P,Q; w is K,C,T,R,S.  Tap (t, r, s)
 * reads the input at (z*sd - pd + t*dd, p*sh - ph + r*dh, q*sw - pw + s*dw);
 * reads outside the input are zero.
 *
 * Every result is the literal definition summed in fp64, one output element
 * at a time (gather form), threads split only over output elements.
 *
 * Parity status: pinned by tests/test_oracle_pins_3d.py -- depth-1 problems
 * equal the 2-D oracle, depth-only problems equal a 1-D cross-correlation run
 * through the 2-D oracle, every problem equals the sum over depth taps of 2-D
 * convolutions of depth slices, the adjoint identity across the three ops,
 * hand-counted all-ones values, and a library witness.  NaN/Inf propagation
 * is parity unpinned.
 */
#include <stdint.h>

#define IDX5(a, b, c, d, e, B, C, D, E) (((((int64_t)(a) * (B) + (b)) * (C) + (c)) * (D) + (d)) * (E) + (e))

typedef struct {
    int N, C, D, H, W, K, T, R, S;
    int pd, ph, pw, sd, sh, sw, dd, dh, dw;
    int Z, P, Q;
} geom3;

static geom3 make_geom(const int *g)
{
    geom3 q;
    q.N = g[0]; q.C = g[1]; q.D = g[2]; q.H = g[3]; q.W = g[4];
    q.K = g[5]; q.T = g[6]; q.R = g[7]; q.S = g[8];
    q.pd = g[9]; q.ph = g[10]; q.pw = g[11];
    q.sd = g[12]; q.sh = g[13]; q.sw = g[14];
    q.dd = g[15]; q.dh = g[16]; q.dw = g[17];
    q.Z = g[18]; q.P = g[19]; q.Q = g[20];
    return q;
}

/* Zero-padded read of x[n,c,z,h,w]. */
static inline double xpad3(const double *x, const geom3 *g, int n, int c, int z, int h, int w)
{
    if (z < 0 || z >= g->D || h < 0 || h >= g->H || w < 0 || w >= g->W)
        return 0.0;
    return x[IDX5(n, c, z, h, w, g->C, g->D, g->H, g->W)];
}

/* Forward: y[n,k,z,p,q] = sum_{c,t,r,s} X(n, c, z*sd-pd+t*dd, p*sh-ph+r*dh, q*sw-pw+s*dw) * w[k,c,t,r,s]. */
static double fwd3_one(const double *x, const double *w, const geom3 *g, int n, int k, int z, int p, int q)
{
    double acc = 0.0;
    for (int c = 0; c < g->C; ++c)
        for (int t = 0; t < g->T; ++t)
            for (int r = 0; r < g->R; ++r)
                for (int s = 0; s < g->S; ++s)
                    acc += xpad3(x, g, n, c, z * g->sd - g->pd + t * g->dd, p * g->sh - g->ph + r * g->dh,
                                 q * g->sw - g->pw + s * g->dw) *
                           w[IDX5(k, c, t, r, s, g->C, g->T, g->R, g->S)];
    return acc;
}

void oracle_conv3d_fwd(const double *x, const double *w, double *y, const int *dims)
{
    const geom3 g = make_geom(dims);
#pragma omp parallel for collapse(2) schedule(static)
    for (int n = 0; n < g.N; ++n)
        for (int k = 0; k < g.K; ++k)
            for (int z = 0; z < g.Z; ++z)
                for (int p = 0; p < g.P; ++p)
                    for (int q = 0; q < g.Q; ++q)
                        y[IDX5(n, k, z, p, q, g.K, g.Z, g.P, g.Q)] = fwd3_one(x, w, &g, n, k, z, p, q);
}

/* The output index along one dim that reads input index i through tap u:
 * i = o*stride - pad + u*dil, so o = (i + pad - u*dil) / stride when that
 * quotient is a whole number in [0, O).  Returns -1 when no output reads it.
 * The sign test comes before the divisibility test so that C's truncating %
 * never sees a negative operand. */
static inline int reader(int i, int u, int pad, int stride, int dil, int O)
{
    int t = i + pad - u * dil;
    if (t < 0 || t % stride != 0)
        return -1;
    int o = t / stride;
    return o < O ? o : -1;
}

/* Backward data: dx[n,c,z,h,w] = sum over (k,t,r,s) of dy[n,k,oz,oh,ow] * w[k,c,t,r,s]
 * over the output positions (oz,oh,ow) whose tap (t,r,s) reads (z,h,w). */
static double bwd_data3_one(const double *dy, const double *w, const geom3 *g, int n, int c, int z, int h,
                            int ww)
{
    double acc = 0.0;
    for (int k = 0; k < g->K; ++k)
        for (int t = 0; t < g->T; ++t) {
            int oz = reader(z, t, g->pd, g->sd, g->dd, g->Z);
            if (oz < 0)
                continue;
            for (int r = 0; r < g->R; ++r) {
                int oh = reader(h, r, g->ph, g->sh, g->dh, g->P);
                if (oh < 0)
                    continue;
                for (int s = 0; s < g->S; ++s) {
                    int ow = reader(ww, s, g->pw, g->sw, g->dw, g->Q);
                    if (ow < 0)
                        continue;
                    acc += dy[IDX5(n, k, oz, oh, ow, g->K, g->Z, g->P, g->Q)] *
                           w[IDX5(k, c, t, r, s, g->C, g->T, g->R, g->S)];
                }
            }
        }
    return acc;
}

void oracle_conv3d_bwd_data(const double *dy, const double *w, double *dx, const int *dims)
{
    const geom3 g = make_geom(dims);
#pragma omp parallel for collapse(2) schedule(static)
    for (int n = 0; n < g.N; ++n)
        for (int c = 0; c < g.C; ++c)
            for (int z = 0; z < g.D; ++z)
                for (int h = 0; h < g.H; ++h)
                    for (int ww = 0; ww < g.W; ++ww)
                        dx[IDX5(n, c, z, h, ww, g.C, g.D, g.H, g.W)] = bwd_data3_one(dy, w, &g, n, c, z, h, ww);
}

/* Backward filter: dw[k,c,t,r,s] = sum_{n,z,p,q} X(n, c, z*sd-pd+t*dd, p*sh-ph+r*dh, q*sw-pw+s*dw) * dy[n,k,z,p,q]. */
static double bwd_filter3_one(const double *x, const double *dy, const geom3 *g, int k, int c, int t, int r,
                              int s)
{
    double acc = 0.0;
    for (int n = 0; n < g->N; ++n)
        for (int z = 0; z < g->Z; ++z)
            for (int p = 0; p < g->P; ++p)
                for (int q = 0; q < g->Q; ++q)
                    acc += xpad3(x, g, n, c, z * g->sd - g->pd + t * g->dd, p * g->sh - g->ph + r * g->dh,
                                 q * g->sw - g->pw + s * g->dw) *
                           dy[IDX5(n, k, z, p, q, g->K, g->Z, g->P, g->Q)];
    return acc;
}

void oracle_conv3d_bwd_filter(const double *x, const double *dy, double *dw, const int *dims)
{
    const geom3 g = make_geom(dims);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int k = 0; k < g.K; ++k)
        for (int c = 0; c < g.C; ++c)
            for (int t = 0; t < g.T; ++t)
                for (int r = 0; r < g.R; ++r)
                    for (int s = 0; s < g.S; ++s)
                        dw[IDX5(k, c, t, r, s, g.C, g.T, g.R, g.S)] = bwd_filter3_one(x, dy, &g, k, c, t, r, s);
}

/* Sampled evaluation: the same per-element definitions at the flat output indices
 * idx[0..count) (y / dx / dw in their NCDHW / KCTRS order), for parity at full sizes. */
void oracle_conv3d_fwd_at(const double *x, const double *w, const int *dims, const int64_t *idx, int64_t count,
                          double *out)
{
    const geom3 g = make_geom(dims);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; ++i) {
        int64_t f = idx[i];
        const int q = (int)(f % g.Q); f /= g.Q;
        const int p = (int)(f % g.P); f /= g.P;
        const int z = (int)(f % g.Z); f /= g.Z;
        const int k = (int)(f % g.K); f /= g.K;
        out[i] = fwd3_one(x, w, &g, (int)f, k, z, p, q);
    }
}

void oracle_conv3d_bwd_data_at(const double *dy, const double *w, const int *dims, const int64_t *idx,
                               int64_t count, double *out)
{
    const geom3 g = make_geom(dims);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; ++i) {
        int64_t f = idx[i];
        const int ww = (int)(f % g.W); f /= g.W;
        const int h = (int)(f % g.H); f /= g.H;
        const int z = (int)(f % g.D); f /= g.D;
        const int c = (int)(f % g.C); f /= g.C;
        out[i] = bwd_data3_one(dy, w, &g, (int)f, c, z, h, ww);
    }
}

void oracle_conv3d_bwd_filter_at(const double *x, const double *dy, const int *dims, const int64_t *idx,
                                 int64_t count, double *out)
{
    const geom3 g = make_geom(dims);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < count; ++i) {
        int64_t f = idx[i];
        const int s = (int)(f % g.S); f /= g.S;
        const int r = (int)(f % g.R); f /= g.R;
        const int t = (int)(f % g.T); f /= g.T;
        const int c = (int)(f % g.C); f /= g.C;
        out[i] = bwd_filter3_one(x, dy, &g, (int)f, c, t, r, s);
    }
}

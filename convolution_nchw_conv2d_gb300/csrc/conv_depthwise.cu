// conv_depthwise.cu -- depthwise convolution (groups == C: one input channel per group), the
// three ops as direct sums on CUDA cores (see DwPlan).  A depthwise layer is a grouped
// convolution whose groups each have one input channel (Apache MXNet mkldnn_deconvolution.cc,
// DeconvDescCreator: num_group; the grouped filter is K x C/groups x R x S); its GEMM view has
// N = K / C columns per group, far too narrow for the tensor cores, and the layer is memory
// bound.  A block takes units of one plane's band of rows: it stages the band's zero-padded
// input window in shared memory (eight loads in flight per thread), then each output element is
// one thread's fixed-order fp32 sum over its taps (forward, backward-data at unit stride), or
// each thread keeps every tap's running sum of x * dy in registers (filter gradient, reduced per
// block and then over image splits in a fixed order).  3x3, 5x5 and 7x7 filters are compiled
// with their taps and band offsets in registers; rows too wide to stage and strided
// backward-data read global memory directly.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <type_traits>

#include "conv_plan.h"
#include "launch_util.cuh"

namespace cg3 {

namespace {

template <int DT>
__device__ __forceinline__ float ld(const void* base, long long i) {
  if constexpr (DT == 0)
    return __ldg(static_cast<const float*>(base) + i);
  else
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
}

template <int DT>
__device__ __forceinline__ float ld_rw(const void* base, long long i) {  // a location this grid writes
  if constexpr (DT == 0)
    return static_cast<const float*>(base)[i];
  else
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
}

template <int DT>
__device__ __forceinline__ void st(void* base, long long i, float v) {
  if constexpr (DT == 0)
    static_cast<float*>(base)[i] = v;
  else
    static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
}

// Filter element of tap (r, s) of output channel k (the filter is K x 1 x R x S).
__device__ __forceinline__ long long wtap(const DwPlan& p, int k, int r, int s) {
  if (p.flip) {
    r = p.R - 1 - r;
    s = p.S - 1 - s;
  }
  return ((long long)k * p.R + r) * p.S + s;
}

// Stages the window of nrows x wt elements into dst (row-major): element (row, col) is the
// global element at index at(row, col), or 0 where at() returns a negative index.  Each thread
// takes elements tid, tid + blockDim, ... and keeps kDwLoads of its loads in flight before
// storing them; the (row, col) of its next element advances by blockDim without a division.
constexpr int kDwLoads = 8;
template <int DT, class At>
__device__ __forceinline__ void stage_window(float* dst, const void* src, int nrows, int wt, At at) {
  const int total = nrows * wt;
  const int step = (int)blockDim.x;
  const int dq = step / wt, dr = step - dq * wt;
  int row = (int)threadIdx.x / wt, col = (int)threadIdx.x - row * wt;
  for (int e0 = (int)threadIdx.x; e0 < total; e0 += kDwLoads * step) {
    float v[kDwLoads];
#pragma unroll
    for (int u = 0; u < kDwLoads; ++u) {
      const long long gi = e0 + u * step < total ? at(row, col) : -1;
      v[u] = gi >= 0 ? ld<DT>(src, gi) : 0.f;
      row += dq;
      col += dr;
      if (col >= wt) {
        col -= wt;
        ++row;
      }
    }
#pragma unroll
    for (int u = 0; u < kDwLoads; ++u)
      if (e0 + u * step < total) dst[e0 + u * step] = v[u];
  }
}

}  // namespace

constexpr int kDwTile = 1024;  // output positions of one plane per work unit (4 per thread)
constexpr int kDwRun = 4;      // consecutive outputs of a row per thread (staged 3x3 / 5x5 / 7x7)
constexpr int kDwSmem = 16 * 1024;  // bytes of one staged input band (fp32)

// Rows of a forward unit's band (band_rows(p) output rows of one plane) and the staged input
// band's row width: columns iw = col - pw for col < wt, so that output column q, tap s reads col
// q*sw + s*dw.
__host__ __device__ inline int dw_fwd_wt(const DwPlan& p) { return (p.Q - 1) * p.sw + (p.S - 1) * p.dw + 1; }
__host__ __device__ inline int dw_fwd_in_rows(const DwPlan& p, int bp) { return (bp - 1) * p.sh + (p.R - 1) * p.dh + 1; }
__host__ inline int dw_fwd_band(const DwPlan& p) {
  int bp = p.P;
  while (bp > 1 && (long long)dw_fwd_in_rows(p, bp) * dw_fwd_wt(p) * 4 > kDwSmem) bp = (bp + 1) / 2;
  return bp;
}

// Forward: a unit is a band of bp output rows of one plane (n, k).  The block stages the band's
// input rows of channel k / M (zero outside x, so the sums need no bounds checks) and the
// filter's taps in shared memory, then each thread sums the taps of its outputs (consecutive
// threads on consecutive q: conflict-free shared reads at unit stride, coalesced y writes).
// RT x ST > 0: the filter size at compile time (taps and their band offsets in registers,
// the tap loop unrolled); 0 x 0: any size.
template <int DT, int RT, int ST>
__global__ void __launch_bounds__(256) dw_fwd_kernel(const __grid_constant__ DwPlan p, int bp) {
  extern __shared__ float dw_smem[];
  const int PQ = p.P * p.Q;
  const int wt = dw_fwd_wt(p), nrows = dw_fwd_in_rows(p, bp);
  const int RS = p.R * p.S;
  float* taps = dw_smem;                  // R*S filter taps (in the order the sums read them)
  float* band = dw_smem + ((RS + 3) & ~3);  // nrows x wt staged input
  const int nb = (p.P + bp - 1) / bp;     // bands per plane
  const long long units = (long long)p.N * p.K * nb;
  for (long long u = blockIdx.x; u < units; u += gridDim.x) {
    const long long nk = u / nb;
    const int b = (int)(u - nk * nb);
    const int k = (int)(nk % p.K);
    const long long n = nk / p.K;
    const int c = k / p.M;
    const int p0 = b * bp, np = min(bp, p.P - p0);
    const int ih0 = p0 * p.sh - p.ph;
    const long long xb = (n * p.C + c) * (long long)p.H * p.W;
    __syncthreads();  // the previous unit's reads of the band are done
    for (int t = (int)threadIdx.x; t < RS; t += (int)blockDim.x) taps[t] = ld<DT>(p.w, wtap(p, k, t / p.S, t % p.S));
    const int rows_used = (np - 1) * p.sh + (p.R - 1) * p.dh + 1;
    stage_window<DT>(band, p.x, rows_used, wt, [&](int row, int col) -> long long {
      const int ih = ih0 + row, iw = col - p.pw;
      return (ih >= 0 && ih < p.H && iw >= 0 && iw < p.W) ? xb + (long long)ih * p.W + iw : -1;
    });
    __syncthreads();
    const long long yb = nk * PQ + (long long)p0 * p.Q;
    if constexpr (RT > 0 && ST > 0) {
      float tv[RT * ST];
      int toff[RT * ST];
#pragma unroll
      for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int s = 0; s < ST; ++s) {
          tv[r * ST + s] = taps[r * ST + s];
          toff[r * ST + s] = r * p.dh * wt + s * p.dw;
        }
      const float bv = p.bias != nullptr ? ld<DT>(p.bias, k) : 0.f;
      if (p.sw == 1 && p.dw == 1) {
        // kDwRun consecutive outputs of a row per thread: each band row's kDwRun + ST - 1 inputs
        // are read once for all of them (the reads past a row's end, at most kDwRun - 1 into the
        // next row or the band's padding, only feed outputs past Q, which are not stored)
        const int nq = (p.Q + kDwRun - 1) / kDwRun;
        for (int it = (int)threadIdx.x; it < np * nq; it += (int)blockDim.x) {
          const int pp = it / nq, q0 = (it - pp * nq) * kDwRun;
          float acc[kDwRun];
#pragma unroll
          for (int j = 0; j < kDwRun; ++j) acc[j] = 0.f;
#pragma unroll
          for (int r = 0; r < RT; ++r) {
            const float* row = band + (pp * p.sh + r * p.dh) * wt + q0;
            float v[kDwRun + ST - 1];
#pragma unroll
            for (int i = 0; i < kDwRun + ST - 1; ++i) v[i] = row[i];
#pragma unroll
            for (int ss = 0; ss < ST; ++ss)
#pragma unroll
              for (int j = 0; j < kDwRun; ++j) acc[j] = fmaf(v[j + ss], tv[r * ST + ss], acc[j]);
          }
#pragma unroll
          for (int j = 0; j < kDwRun; ++j) {
            if (q0 + j < p.Q) {
              const long long o = yb + (long long)pp * p.Q + q0 + j;
              float a = acc[j] + bv;
              if (p.beta != 0.f) a += p.beta * ld_rw<DT>(p.out, o);
              st<DT>(p.out, o, a);
            }
          }
        }
        continue;
      }
      for (int o = (int)threadIdx.x; o < np * p.Q; o += (int)blockDim.x) {
        const int pp = o / p.Q, q = o - pp * p.Q;
        const float* src = band + pp * p.sh * wt + q * p.sw;
        float acc = 0.f;
#pragma unroll
        for (int t = 0; t < RT * ST; ++t) acc = fmaf(src[toff[t]], tv[t], acc);
        acc += bv;
        if (p.beta != 0.f) acc += p.beta * ld_rw<DT>(p.out, yb + o);
        st<DT>(p.out, yb + o, acc);
      }
      continue;
    }
    for (int o = (int)threadIdx.x; o < np * p.Q; o += (int)blockDim.x) {
      const int pp = o / p.Q, q = o - pp * p.Q;
      const float* src = band + pp * p.sh * wt + q * p.sw;
      float acc = 0.f;
      for (int r = 0; r < p.R; ++r)
        for (int s = 0; s < p.S; ++s) acc = fmaf(src[r * p.dh * wt + s * p.dw], taps[r * p.S + s], acc);
      if (p.bias != nullptr) acc += ld<DT>(p.bias, k);
      if (p.beta != 0.f) acc += p.beta * ld_rw<DT>(p.out, yb + o);
      st<DT>(p.out, yb + o, acc);
    }
  }
}

// Forward without staging (a band row wider than the staging limit): work units of kDwTile
// positions of one output plane (n, k); thread t takes positions
// t, t + 256, ... of the unit (consecutive threads on consecutive q: coalesced x reads and y
// writes); the plane's indices are computed once per unit, positions in 32 bits.
template <int DT>
__global__ void __launch_bounds__(256) dw_fwd_direct_kernel(const __grid_constant__ DwPlan p) {
  const int PQ = p.P * p.Q;
  const int tpp = (PQ + kDwTile - 1) / kDwTile;  // units per plane
  const long long units = (long long)p.N * p.K * tpp;
  for (long long u = blockIdx.x; u < units; u += gridDim.x) {
    const long long nk = u / tpp;
    const int tile = (int)(u - nk * tpp);
    const int k = (int)(nk % p.K);
    const long long n = nk / p.K;
    const int c = k / p.M;
    const long long xb = (n * p.C + c) * (long long)p.H * p.W;
    const long long yb = nk * PQ;
#pragma unroll
    for (int j = 0; j < kDwTile / 256; ++j) {
      const int pos = tile * kDwTile + j * 256 + (int)threadIdx.x;
      if (pos >= PQ) break;
      const int pp = pos / p.Q, q = pos - pp * p.Q;
      float acc = 0.f;
      for (int r = 0; r < p.R; ++r) {
        const int ih = pp * p.sh - p.ph + r * p.dh;
        if (ih < 0 || ih >= p.H) continue;
        for (int s = 0; s < p.S; ++s) {
          const int iw = q * p.sw - p.pw + s * p.dw;
          if (iw < 0 || iw >= p.W) continue;
          acc = fmaf(ld<DT>(p.x, xb + (long long)ih * p.W + iw), ld<DT>(p.w, wtap(p, k, r, s)), acc);
        }
      }
      if (p.bias != nullptr) acc += ld<DT>(p.bias, k);
      if (p.beta != 0.f) acc += p.beta * ld_rw<DT>(p.out, yb + pos);
      st<DT>(p.out, yb + pos, acc);
    }
  }
}

// Backward-data: work units of kDwTile positions of one dx plane (n, c); each dx element sums
// the output channels c*M .. c*M + M - 1 and the taps that reach it, in the order (m, r, s).
template <int DT>
__global__ void __launch_bounds__(256) dw_bwd_data_kernel(const __grid_constant__ DwPlan p) {
  const int HW = p.H * p.W;
  const long long PQ = (long long)p.P * p.Q;
  const int tpp = (HW + kDwTile - 1) / kDwTile;
  const long long units = (long long)p.N * p.C * tpp;
  for (long long u = blockIdx.x; u < units; u += gridDim.x) {
    const long long nc = u / tpp;
    const int tile = (int)(u - nc * tpp);
    const int c = (int)(nc % p.C);
    const long long n = nc / p.C;
#pragma unroll
    for (int j = 0; j < kDwTile / 256; ++j) {
      const int pos = tile * kDwTile + j * 256 + (int)threadIdx.x;
      if (pos >= HW) break;
      const int h = pos / p.W, w = pos - h * p.W;
      float acc = 0.f;
      for (int m = 0; m < p.M; ++m) {
        const int k = c * p.M + m;
        const long long db = (n * p.K + k) * PQ;
        for (int r = 0; r < p.R; ++r) {
          const int th = h + p.ph - r * p.dh;  // = pp * sh for the dy row pp it reaches
          if (th < 0 || th % p.sh != 0) continue;
          const int pp = th / p.sh;
          if (pp >= p.P) continue;
          for (int s = 0; s < p.S; ++s) {
            const int tw = w + p.pw - s * p.dw;
            if (tw < 0 || tw % p.sw != 0) continue;
            const int q = tw / p.sw;
            if (q >= p.Q) continue;
            acc = fmaf(ld<DT>(p.dy, db + (long long)pp * p.Q + q), ld<DT>(p.w, wtap(p, k, r, s)), acc);
          }
        }
      }
      const long long o = nc * HW + pos;
      if (p.bias != nullptr) acc += ld<DT>(p.bias, c);
      if (p.beta != 0.f) acc += p.beta * ld_rw<DT>(p.out, o);
      st<DT>(p.out, o, acc);
    }
  }
}

// Backward-data at unit stride: a unit is a band of bh rows of one dx plane (n, c).  The block
// stages, for each of the channel's M output channels, the dy rows the band reads (dy row
// h + ph - r*dh, zero outside dy) with columns w + pw - s*dw for col = w + (S-1)*dw - s*dw, and
// the filter taps; each thread then sums, for each of its dx elements, the taps in the order
// (m, r, s).
__host__ __device__ inline int dw_bd_wt(const DwPlan& p) { return p.W + (p.S - 1) * p.dw; }
__host__ __device__ inline int dw_bd_rows(const DwPlan& p, int bh) { return bh + (p.R - 1) * p.dh; }
__host__ inline int dw_bd_band(const DwPlan& p) {
  int bh = p.H;
  while (bh > 1 && (long long)p.M * dw_bd_rows(p, bh) * dw_bd_wt(p) * 4 > kDwSmem) bh = (bh + 1) / 2;
  return bh;
}

template <int DT, int RT, int ST>
__global__ void __launch_bounds__(256) dw_bwd_data_s1_kernel(const __grid_constant__ DwPlan p, int bh) {
  extern __shared__ float dw_smem[];
  const int HW = p.H * p.W;
  const long long PQ = (long long)p.P * p.Q;
  const int wt = dw_bd_wt(p), nrows = dw_bd_rows(p, bh);
  const int RS = p.R * p.S;
  float* taps = dw_smem;                        // M x R*S
  float* band = dw_smem + ((p.M * RS + 3) & ~3);  // M x nrows x wt
  const int nb = (p.H + bh - 1) / bh;
  const long long units = (long long)p.N * p.C * nb;
  for (long long u = blockIdx.x; u < units; u += gridDim.x) {
    const long long nc = u / nb;
    const int b = (int)(u - nc * nb);
    const int c = (int)(nc % p.C);
    const long long n = nc / p.C;
    const int h0 = b * bh, nh = min(bh, p.H - h0);
    const int rows_used = nh + (p.R - 1) * p.dh;
    const int pr0 = h0 + p.ph - (p.R - 1) * p.dh;  // dy row of staged row 0
    const int qc0 = p.pw - (p.S - 1) * p.dw;       // dy column of staged column 0
    __syncthreads();
    for (int t = (int)threadIdx.x; t < p.M * RS; t += (int)blockDim.x) {
      const int m = t / RS, rs = t - m * RS;
      taps[t] = ld<DT>(p.w, wtap(p, c * p.M + m, rs / p.S, rs % p.S));
    }
    for (int m = 0; m < p.M; ++m) {
      const long long db = (n * p.K + c * p.M + m) * PQ;
      float* bm = band + m * nrows * wt;
      stage_window<DT>(bm, p.dy, rows_used, wt, [&](int row, int col) -> long long {
        const int pp = pr0 + row, q = qc0 + col;
        return (pp >= 0 && pp < p.P && q >= 0 && q < p.Q) ? db + (long long)pp * p.Q + q : -1;
      });
    }
    __syncthreads();
    const long long ob = nc * HW + (long long)h0 * p.W;
    if constexpr (RT > 0 && ST > 0) {
      if (p.M == 1) {  // one output channel per input channel: taps and offsets in registers
        float tv[RT * ST];
        int toff[RT * ST];
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
          for (int s = 0; s < ST; ++s) {
            tv[r * ST + s] = taps[r * ST + s];
            toff[r * ST + s] = -(r * p.dh) * wt - s * p.dw;
          }
        const float bv = p.bias != nullptr ? ld<DT>(p.bias, c) : 0.f;
        if (p.dw == 1) {
          // kDwRun consecutive dx elements of a row per thread (as the forward does): output
          // w0 + j, tap s reads staged column w0 + j + ST - 1 - s
          const int nw = (p.W + kDwRun - 1) / kDwRun;
          for (int it = (int)threadIdx.x; it < nh * nw; it += (int)blockDim.x) {
            const int hh = it / nw, w0 = (it - hh * nw) * kDwRun;
            float acc[kDwRun];
#pragma unroll
            for (int j = 0; j < kDwRun; ++j) acc[j] = 0.f;
#pragma unroll
            for (int r = 0; r < RT; ++r) {
              const float* row = band + (hh + (RT - 1 - r) * p.dh) * wt + w0;
              float v[kDwRun + ST - 1];
#pragma unroll
              for (int i = 0; i < kDwRun + ST - 1; ++i) v[i] = row[i];
#pragma unroll
              for (int ss = 0; ss < ST; ++ss)
#pragma unroll
                for (int j = 0; j < kDwRun; ++j) acc[j] = fmaf(v[j + ST - 1 - ss], tv[r * ST + ss], acc[j]);
            }
#pragma unroll
            for (int j = 0; j < kDwRun; ++j) {
              if (w0 + j < p.W) {
                const long long o = ob + (long long)hh * p.W + w0 + j;
                float a = acc[j] + bv;
                if (p.beta != 0.f) a += p.beta * ld_rw<DT>(p.out, o);
                st<DT>(p.out, o, a);
              }
            }
          }
          continue;
        }
        for (int o = (int)threadIdx.x; o < nh * p.W; o += (int)blockDim.x) {
          const int hh = o / p.W, w = o - hh * p.W;
          const float* bm = band + (hh + (RT - 1) * p.dh) * wt + w + (ST - 1) * p.dw;
          float acc = 0.f;
#pragma unroll
          for (int t = 0; t < RT * ST; ++t) acc = fmaf(bm[toff[t]], tv[t], acc);
          acc += bv;
          if (p.beta != 0.f) acc += p.beta * ld_rw<DT>(p.out, ob + o);
          st<DT>(p.out, ob + o, acc);
        }
        continue;
      }
    }
    for (int o = (int)threadIdx.x; o < nh * p.W; o += (int)blockDim.x) {
      const int hh = o / p.W, w = o - hh * p.W;
      float acc = 0.f;
      for (int m = 0; m < p.M; ++m) {
        const float* bm = band + m * nrows * wt + (hh + (p.R - 1) * p.dh) * wt + w + (p.S - 1) * p.dw;
        const float* tm = taps + m * RS;
        for (int r = 0; r < p.R; ++r)
          for (int s = 0; s < p.S; ++s) acc = fmaf(bm[-(r * p.dh) * wt - s * p.dw], tm[r * p.S + s], acc);
      }
      if (p.bias != nullptr) acc += ld<DT>(p.bias, c);
      if (p.beta != 0.f) acc += p.beta * ld_rw<DT>(p.out, ob + o);
      st<DT>(p.out, ob + o, acc);
    }
  }
}

// Backward-filter partials: block (k, split) sums, for every tap (r, s) in turn, x * dy over the
// positions (p, q) of its split's images, each thread a strided subset in increasing order, then
// a fixed-order tree over the block: partial[(split * K + k) * R*S + r*S + s].
template <int DT>
__global__ void __launch_bounds__(256) dw_wgrad_kernel(const __grid_constant__ DwPlan p) {
  __shared__ float red[256];
  const int k = (int)(blockIdx.x % p.K);
  const int sp = (int)(blockIdx.x / p.K);
  const int c = k / p.M;
  const int PQ = p.P * p.Q;
  const int n0 = sp * p.n_per_split, n1 = min(p.N, n0 + p.n_per_split);
  for (int r = 0; r < p.R; ++r)
    for (int s = 0; s < p.S; ++s) {
      float acc = 0.f;
      for (int n = n0; n < n1; ++n) {
        const long long xb = ((long long)n * p.C + c) * p.H * p.W;
        const long long db = ((long long)n * p.K + k) * PQ;
        for (int pos = (int)threadIdx.x; pos < PQ; pos += (int)blockDim.x) {
          const int pp = pos / p.Q, q = pos - pp * p.Q;
          const int ih = pp * p.sh - p.ph + r * p.dh, iw = q * p.sw - p.pw + s * p.dw;
          if (ih < 0 || ih >= p.H || iw < 0 || iw >= p.W) continue;
          acc = fmaf(ld<DT>(p.x, xb + (long long)ih * p.W + iw), ld<DT>(p.dy, db + pos), acc);
        }
      }
      red[threadIdx.x] = acc;
      __syncthreads();
      for (int h = 128; h > 0; h >>= 1) {
        if ((int)threadIdx.x < h) red[threadIdx.x] += red[threadIdx.x + h];
        __syncthreads();
      }
      if (threadIdx.x == 0) p.partial[((long long)sp * p.K + k) * p.R * p.S + r * p.S + s] = red[0];
      __syncthreads();
    }
}

// Backward-filter partials, staged: block (k, split) walks its images' output-row bands (the
// forward's bands): the block stages the band's x rows (zero outside x, as the forward does) and
// dy rows in shared memory, then each thread adds, for each of its outputs o in increasing
// order, dy[o] times the band's input under every tap into its RSM register accumulators (R*S
// <= RSM); a fixed-order tree over the block per tap gives the split's partials.
template <int DT, int RSM, int RT, int ST>
__global__ void __launch_bounds__(256) dw_wgrad_band_kernel(const __grid_constant__ DwPlan p, int bp) {
  extern __shared__ float dw_smem[];
  const int k = (int)(blockIdx.x % p.K);
  const int sp = (int)(blockIdx.x / p.K);
  const int c = k / p.M;
  const int PQ = p.P * p.Q;
  const int wt = dw_fwd_wt(p), nrows = dw_fwd_in_rows(p, bp);
  const int RS = p.R * p.S;
  float* band = dw_smem;                 // nrows x wt staged x
  float* dyb = dw_smem + nrows * wt;     // bp x Q staged dy
  float acc[RSM];
#pragma unroll
  for (int t = 0; t < RSM; ++t) acc[t] = 0.f;
  const int n0 = sp * p.n_per_split, n1 = min(p.N, n0 + p.n_per_split);
  for (int n = n0; n < n1; ++n) {
    const long long xb = ((long long)n * p.C + c) * p.H * p.W;
    const long long db = ((long long)n * p.K + k) * PQ;
    for (int p0 = 0; p0 < p.P; p0 += bp) {
      const int np = min(bp, p.P - p0);
      const int ih0 = p0 * p.sh - p.ph;
      const int rows_used = (np - 1) * p.sh + (p.R - 1) * p.dh + 1;
      __syncthreads();  // the previous band's reads are done
      stage_window<DT>(band, p.x, rows_used, wt, [&](int row, int col) -> long long {
        const int ih = ih0 + row, iw = col - p.pw;
        return (ih >= 0 && ih < p.H && iw >= 0 && iw < p.W) ? xb + (long long)ih * p.W + iw : -1;
      });
      stage_window<DT>(dyb, p.dy, np, p.Q, [&](int row, int col) -> long long {
        return db + (long long)(p0 + row) * p.Q + col;
      });
      __syncthreads();
      if constexpr (RT > 0 && ST > 0) {  // RSM == RT * ST: every tap's offset in a register
        if (p.sw == 1 && p.dw == 1) {
          // kDwRun consecutive outputs of a row per thread: each band row's kDwRun + ST - 1 inputs
          // read once (columns past the row's end read as 0; outputs past Q carry dy = 0)
          const int nq = (p.Q + kDwRun - 1) / kDwRun;
          for (int it = (int)threadIdx.x; it < np * nq; it += (int)blockDim.x) {
            const int pp = it / nq, q0 = (it - pp * nq) * kDwRun;
            float g[kDwRun];
#pragma unroll
            for (int j = 0; j < kDwRun; ++j) g[j] = q0 + j < p.Q ? dyb[pp * p.Q + q0 + j] : 0.f;
#pragma unroll
            for (int r = 0; r < RT; ++r) {
              const float* row = band + (pp * p.sh + r * p.dh) * wt + q0;
              float v[kDwRun + ST - 1];
#pragma unroll
              for (int i = 0; i < kDwRun + ST - 1; ++i) v[i] = q0 + i < wt ? row[i] : 0.f;
#pragma unroll
              for (int ss = 0; ss < ST; ++ss)
#pragma unroll
                for (int j = 0; j < kDwRun; ++j) acc[r * ST + ss] = fmaf(v[j + ss], g[j], acc[r * ST + ss]);
            }
          }
          continue;
        }
        int toff[RT * ST];
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
          for (int s = 0; s < ST; ++s) toff[r * ST + s] = r * p.dh * wt + s * p.dw;
        for (int o = (int)threadIdx.x; o < np * p.Q; o += (int)blockDim.x) {
          const int pp = o / p.Q, q = o - pp * p.Q;
          const float g = dyb[o];
          const float* src = band + pp * p.sh * wt + q * p.sw;
#pragma unroll
          for (int t = 0; t < RT * ST; ++t) acc[t] = fmaf(src[toff[t]], g, acc[t]);
        }
      } else {
        for (int o = (int)threadIdx.x; o < np * p.Q; o += (int)blockDim.x) {
          const int pp = o / p.Q, q = o - pp * p.Q;
          const float g = dyb[o];
          const float* src = band + pp * p.sh * wt + q * p.sw;
#pragma unroll
          for (int t = 0; t < RSM; ++t) {
            if (t < RS) {
              const int r = t / p.S, s = t - r * p.S;
              acc[t] = fmaf(src[r * p.dh * wt + s * p.dw], g, acc[t]);
            }
          }
        }
      }
    }
  }
  // per tap: a fixed-order tree over the block's threads (the band area is free now)
  float* red = dw_smem;
  for (int t = 0; t < RS && t < RSM; ++t) {
    __syncthreads();
    float v = 0.f;
#pragma unroll
    for (int u = 0; u < RSM; ++u)
      if (u == t) v = acc[u];
    red[threadIdx.x] = v;
    __syncthreads();
    for (int h = 128; h > 0; h >>= 1) {
      if ((int)threadIdx.x < h) red[threadIdx.x] += red[threadIdx.x + h];
      __syncthreads();
    }
    if (threadIdx.x == 0) p.partial[((long long)sp * p.K + k) * RS + t] = red[0];
  }
}

// dw[k, 0, r', s'] = sum over splits, in split order, of the tap's partials (+ beta * dw).
template <int DT>
__global__ void __launch_bounds__(256) dw_wgrad_reduce_kernel(const __grid_constant__ DwPlan p) {
  const int RS = p.R * p.S;
  const long long total = (long long)p.K * RS;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int k = (int)(i / RS), t = (int)(i - (long long)k * RS);
    float v = 0.f;
    for (int sp = 0; sp < p.nsplit; ++sp) v += p.partial[((long long)sp * p.K + k) * RS + t];
    const long long o = wtap(p, k, t / p.S, t % p.S);
    if (p.beta != 0.f) v += p.beta * ld_rw<DT>(p.out, o);
    st<DT>(p.out, o, v);
  }
}

// ---------------------------------------------------------------------------- launchers
// The staged forward and unit-stride backward-data kernels for 3x3, 5x5 and 7x7 filters
// (compile-time sizes) and any other size.
struct KernelFwd {
  template <int DT, int RT, int ST>
  static auto get() { return dw_fwd_kernel<DT, RT, ST>; }
};
struct KernelBwdData {
  template <int DT, int RT, int ST>
  static auto get() { return dw_bwd_data_s1_kernel<DT, RT, ST>; }
};

template <int DT, int RT, int ST, class K>
static cudaError_t launch_sized(const DwPlan& p, unsigned g, int band, size_t smem, cudaStream_t st) {
  static std::atomic<int> set_bytes[kMaxDevices];
  auto kern = K::template get<DT, RT, ST>();
  const cudaError_t e = ensure_dyn_smem(kern, smem, set_bytes);
  if (e != cudaSuccess) return e;
  kern<<<g, 256, smem, st>>>(p, band);
  return cudaGetLastError();
}

template <int DT, class K>
static cudaError_t launch_by_size(const DwPlan& p, K, unsigned g, int band, size_t smem, cudaStream_t st) {
  if (p.R == 3 && p.S == 3) return launch_sized<DT, 3, 3, K>(p, g, band, smem, st);
  if (p.R == 5 && p.S == 5) return launch_sized<DT, 5, 5, K>(p, g, band, smem, st);
  if (p.R == 7 && p.S == 7) return launch_sized<DT, 7, 7, K>(p, g, band, smem, st);
  return launch_sized<DT, 0, 0, K>(p, g, band, smem, st);
}
static unsigned dw_grid(long long total, int num_sms) {
  return (unsigned)std::max(1ll, std::min<long long>((total + 255) / 256, (long long)num_sms * 16));
}

size_t dw_fwd_smem_bytes(const DwPlan& p) {
  const int bp = dw_fwd_band(p);
  // + kDwRun: the reads of a row's last run past the band's end
  return ((size_t)((p.R * p.S + 3) & ~3) + (size_t)dw_fwd_in_rows(p, bp) * dw_fwd_wt(p) + kDwRun) * sizeof(float);
}

cudaError_t launch_dw_fwd(const DwPlan& p, int dt, int num_sms, cudaStream_t st) {
  const int bp = dw_fwd_band(p);
  const size_t smem = dw_fwd_smem_bytes(p);
  if (smem > 4 * (size_t)kDwSmem) {  // one band row past the staging limit: unstaged reads
    const long long tpp = ((long long)p.P * p.Q + kDwTile - 1) / kDwTile;
    const unsigned g = (unsigned)std::max(1ll, std::min<long long>((long long)p.N * p.K * tpp, (long long)num_sms * 8));
    if (dt == 0)
      dw_fwd_direct_kernel<0><<<g, 256, 0, st>>>(p);
    else
      dw_fwd_direct_kernel<1><<<g, 256, 0, st>>>(p);
    return cudaGetLastError();
  }
  const long long units = (long long)p.N * p.K * ((p.P + bp - 1) / bp);
  const unsigned g = (unsigned)std::max(1ll, std::min<long long>(units, (long long)num_sms * 8));
  return dt == 0 ? launch_by_size<0>(p, KernelFwd(), g, bp, smem, st) : launch_by_size<1>(p, KernelFwd(), g, bp, smem, st);
}

size_t dw_bd_smem_bytes(const DwPlan& p) {
  const int bh = dw_bd_band(p);
  return ((size_t)((p.M * p.R * p.S + 3) & ~3) + (size_t)p.M * dw_bd_rows(p, bh) * dw_bd_wt(p) + kDwRun) *
         sizeof(float);
}

cudaError_t launch_dw_bwd_data(const DwPlan& p, int dt, int num_sms, cudaStream_t st) {
  if (p.sh == 1 && p.sw == 1 && dw_bd_smem_bytes(p) <= 4 * (size_t)kDwSmem) {  // staged bands
    const int bh = dw_bd_band(p);
    const size_t smem = dw_bd_smem_bytes(p);
    const long long units = (long long)p.N * p.C * ((p.H + bh - 1) / bh);
    const unsigned g = (unsigned)std::max(1ll, std::min<long long>(units, (long long)num_sms * 8));
    return dt == 0 ? launch_by_size<0>(p, KernelBwdData(), g, bh, smem, st)
                   : launch_by_size<1>(p, KernelBwdData(), g, bh, smem, st);
  }
  const long long tpp = ((long long)p.H * p.W + kDwTile - 1) / kDwTile;
  const unsigned g = (unsigned)std::max(1ll, std::min<long long>((long long)p.N * p.C * tpp, (long long)num_sms * 8));
  if (dt == 0)
    dw_bwd_data_kernel<0><<<g, 256, 0, st>>>(p);
  else
    dw_bwd_data_kernel<1><<<g, 256, 0, st>>>(p);
  return cudaGetLastError();
}

template <int DT, int RSM, int RT, int ST>
static cudaError_t launch_dw_wgrad_band(const DwPlan& p, unsigned blocks, int bp, size_t smem, cudaStream_t st) {
  static std::atomic<int> set_bytes[kMaxDevices];
  const cudaError_t e = ensure_dyn_smem(dw_wgrad_band_kernel<DT, RSM, RT, ST>, smem, set_bytes);
  if (e != cudaSuccess) return e;
  dw_wgrad_band_kernel<DT, RSM, RT, ST><<<blocks, 256, smem, st>>>(p, bp);
  return cudaGetLastError();
}

template <int DT>
static cudaError_t launch_dw_wgrad_band_any(const DwPlan& p, unsigned blocks, int bp, size_t smem, cudaStream_t st) {
  const int RS = p.R * p.S;
  if (p.R == 3 && p.S == 3) return launch_dw_wgrad_band<DT, 9, 3, 3>(p, blocks, bp, smem, st);
  if (p.R == 5 && p.S == 5) return launch_dw_wgrad_band<DT, 25, 5, 5>(p, blocks, bp, smem, st);
  if (p.R == 7 && p.S == 7) return launch_dw_wgrad_band<DT, 49, 7, 7>(p, blocks, bp, smem, st);
  return RS <= 9 ? launch_dw_wgrad_band<DT, 9, 0, 0>(p, blocks, bp, smem, st)
                 : RS <= 25 ? launch_dw_wgrad_band<DT, 25, 0, 0>(p, blocks, bp, smem, st)
                            : launch_dw_wgrad_band<DT, 49, 0, 0>(p, blocks, bp, smem, st);
}

// Staged bands with register accumulators for filters of up to 49 taps whose bands fit the
// staging limit; per-tap passes over global memory otherwise.
cudaError_t launch_dw_bwd_filter(const DwPlan& p, int dt, int num_sms, cudaStream_t st) {
  const unsigned blocks = (unsigned)((long long)p.K * p.nsplit);
  const unsigned g = dw_grid((long long)p.K * p.R * p.S, num_sms);
  const int RS = p.R * p.S;
  const int bp = dw_fwd_band(p);
  const size_t smem = std::max<size_t>(256 * sizeof(float),
                                       ((size_t)dw_fwd_in_rows(p, bp) * dw_fwd_wt(p) + (size_t)bp * p.Q) * sizeof(float));
  cudaError_t e = cudaSuccess;
  if (RS <= 49 && smem <= 6 * (size_t)kDwSmem) {
    e = dt == 0 ? launch_dw_wgrad_band_any<0>(p, blocks, bp, smem, st)
                : launch_dw_wgrad_band_any<1>(p, blocks, bp, smem, st);
  } else if (dt == 0) {
    dw_wgrad_kernel<0><<<blocks, 256, 0, st>>>(p);
  } else {
    dw_wgrad_kernel<1><<<blocks, 256, 0, st>>>(p);
  }
  if (e != cudaSuccess) return e;
  if (dt == 0)
    dw_wgrad_reduce_kernel<0><<<g, 256, 0, st>>>(p);
  else
    dw_wgrad_reduce_kernel<1><<<g, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace cg3

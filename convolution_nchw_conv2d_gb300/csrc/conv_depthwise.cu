// conv_depthwise.cu -- depthwise convolution (groups == C: one input channel per group), the
// three ops as direct sums on CUDA cores (see DwPlan).  A depthwise layer is a grouped
// convolution whose groups each have one input channel (Apache MXNet mkldnn_deconvolution.cc,
// DeconvDescCreator: num_group; the grouped filter is K x C/groups x R x S); its GEMM view has
// N = K / C columns per group, far too narrow for the tensor cores, and the layer is memory
// bound, so each output element is one thread's fixed-order sum over its taps.
#include <cuda_bf16.h>

#include <algorithm>
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

}  // namespace

constexpr int kDwTile = 1024;  // output positions of one plane per work unit (4 per thread)

// Forward: work units of kDwTile positions of one output plane (n, k); thread t takes positions
// t, t + 256, ... of the unit (consecutive threads on consecutive q: coalesced x reads and y
// writes); the plane's indices are computed once per unit, positions in 32 bits.
template <int DT>
__global__ void __launch_bounds__(256) dw_fwd_kernel(const __grid_constant__ DwPlan p) {
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
static unsigned dw_grid(long long total, int num_sms) {
  return (unsigned)std::max(1ll, std::min<long long>((total + 255) / 256, (long long)num_sms * 16));
}

cudaError_t launch_dw_fwd(const DwPlan& p, int dt, int num_sms, cudaStream_t st) {
  const long long tpp = ((long long)p.P * p.Q + kDwTile - 1) / kDwTile;
  const unsigned g = (unsigned)std::max(1ll, std::min<long long>((long long)p.N * p.K * tpp, (long long)num_sms * 8));
  if (dt == 0)
    dw_fwd_kernel<0><<<g, 256, 0, st>>>(p);
  else
    dw_fwd_kernel<1><<<g, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_dw_bwd_data(const DwPlan& p, int dt, int num_sms, cudaStream_t st) {
  const long long tpp = ((long long)p.H * p.W + kDwTile - 1) / kDwTile;
  const unsigned g = (unsigned)std::max(1ll, std::min<long long>((long long)p.N * p.C * tpp, (long long)num_sms * 8));
  if (dt == 0)
    dw_bwd_data_kernel<0><<<g, 256, 0, st>>>(p);
  else
    dw_bwd_data_kernel<1><<<g, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_dw_bwd_filter(const DwPlan& p, int dt, int num_sms, cudaStream_t st) {
  const unsigned blocks = (unsigned)((long long)p.K * p.nsplit);
  const unsigned g = dw_grid((long long)p.K * p.R * p.S, num_sms);
  if (dt == 0) {
    dw_wgrad_kernel<0><<<blocks, 256, 0, st>>>(p);
    dw_wgrad_reduce_kernel<0><<<g, 256, 0, st>>>(p);
  } else {
    dw_wgrad_kernel<1><<<blocks, 256, 0, st>>>(p);
    dw_wgrad_reduce_kernel<1><<<g, 256, 0, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace cg3

// conv3d_copy.cu -- layout copies that let the 3-D (NCDHW) operations run as 2-D passes.
//
// A 3-D cross-correlation with T depth taps is the sum over depth taps t of 2-D
// cross-correlations of depth slices: output depth z reads input depth
// d = z*stride_d - pad_d + t*dil_d (zero outside [0, D)).  Gathering, for one t, the slices d(z)
// of every image into a batch of N*Z two-dimensional images makes each depth tap one 2-D problem
// of N*Z images (page "mkldnn_deconvolution.cc": SupportMKLDNNDeconv takes kernels of 1 to 3
// spatial dimensions; DeconvDescCreator takes stride, pad and dilation of the same rank).
// The kernels below are plain element copies (memory-bound, one element per thread iteration,
// coalesced along the innermost H*W run); indices are 64-bit.
#include <cstdint>
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace cg3 {

namespace {

template <int DT>
using Elem = typename std::conditional<DT == 0, float, __nv_bfloat16>::type;

// dst[(n*Zc + z)][c][i] = src[n][c][d][i] with d = z*sd - pd + t*dd, zero outside [0, Dsrc);
// i < HW.  (Identity reshuffle NCDHW -> (N*D)CHW with Zc = Dsrc, sd = 1, pd = 0, t = 0.)
template <int DT>
__global__ void depth_gather_kernel(const Elem<DT>* src, Elem<DT>* dst, int N, int Ch, int Dsrc, long long HW,
                                    int Zc, int sd, int pd, int t, int dd) {
  const long long total = (long long)N * Zc * Ch * HW;
  for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
       o += (long long)gridDim.x * blockDim.x) {
    const long long i = o % HW;
    long long r = o / HW;
    const int c = (int)(r % Ch);
    r /= Ch;
    const int z = (int)(r % Zc);
    const int n = (int)(r / Zc);
    const int d = z * sd - pd + t * dd;
    Elem<DT> v = Elem<DT>(0.f);
    if (d >= 0 && d < Dsrc) v = src[(((long long)n * Ch + c) * Dsrc + d) * HW + i];
    dst[o] = v;
  }
}

// dst[n][c][z][i] = src[(n*Z + z)][c][i]   ((N*Z)CHW -> NCZHW)
template <int DT>
__global__ void batch_to_depth_kernel(const Elem<DT>* src, Elem<DT>* dst, int N, int Ch, int Z, long long HW) {
  const long long total = (long long)N * Ch * Z * HW;
  for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
       o += (long long)gridDim.x * blockDim.x) {
    const long long i = o % HW;
    long long r = o / HW;
    const int z = (int)(r % Z);
    r /= Z;
    const int c = (int)(r % Ch);
    const int n = (int)(r / Ch);
    dst[o] = src[(((long long)n * Z + z) * Ch + c) * HW + i];
  }
}

// acc[n][c][d][i] += src[(n*Z + z)][c][i] for d = z*sd - pd + t*dd inside [0, D): each d gets at
// most one z for a given t, so one launch has no two writers per element.
template <int DT>
__global__ void depth_scatter_add_kernel(const Elem<DT>* src, float* acc, int N, int Ch, int D, long long HW, int Z,
                                         int sd, int pd, int t, int dd) {
  const long long total = (long long)N * Z * Ch * HW;
  for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
       o += (long long)gridDim.x * blockDim.x) {
    const long long i = o % HW;
    long long r = o / HW;
    const int c = (int)(r % Ch);
    r /= Ch;
    const int z = (int)(r % Z);
    const int n = (int)(r / Z);
    const int d = z * sd - pd + t * dd;
    if (d < 0 || d >= D) continue;
    float v;
    if constexpr (DT == 0) v = src[o];
    else v = __bfloat162float(src[o]);
    acc[(((long long)n * Ch + c) * D + d) * HW + i] += v;
  }
}

// dst = acc converted to the tensor type (bf16: round to nearest even)
template <int DT>
__global__ void convert_kernel(const float* acc, Elem<DT>* dst, long long total) {
  for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
       o += (long long)gridDim.x * blockDim.x) {
    if constexpr (DT == 0) dst[o] = acc[o];
    else dst[o] = __float2bfloat16_rn(acc[o]);
  }
}

// One depth tap t of a K x Cg x T x RS filter as a K x Cg x RS filter (to_slice), or back
// (!to_slice: dw[k][c][t][rs] = slice[k][c][rs]).
template <int DT>
__global__ void filter_tap_kernel(const Elem<DT>* src, Elem<DT>* dst, long long KC, int T, int RS, int t, int to_slice) {
  const long long total = KC * RS;
  for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
       o += (long long)gridDim.x * blockDim.x) {
    const long long kc = o / RS;
    const int rs = (int)(o % RS);
    const long long full = (kc * T + t) * RS + rs;
    if (to_slice) dst[o] = src[full];
    else dst[full] = src[o];
  }
}

unsigned grid_for(long long total) {
  const long long b = (total + 255) / 256;
  return (unsigned)(b < 1 ? 1 : (b > 65535 ? 65535 : b));
}

}  // namespace

cudaError_t launch_depth_gather(int dt, const void* src, void* dst, int N, int Ch, int Dsrc, long long HW, int Zc,
                                int sd, int pd, int t, int dd, cudaStream_t st) {
  const unsigned g = grid_for((long long)N * Zc * Ch * HW);
  if (dt == 0)
    depth_gather_kernel<0><<<g, 256, 0, st>>>(static_cast<const float*>(src), static_cast<float*>(dst), N, Ch, Dsrc,
                                               HW, Zc, sd, pd, t, dd);
  else
    depth_gather_kernel<1><<<g, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(src), static_cast<__nv_bfloat16*>(dst),
                                               N, Ch, Dsrc, HW, Zc, sd, pd, t, dd);
  return cudaGetLastError();
}

cudaError_t launch_batch_to_depth(int dt, const void* src, void* dst, int N, int Ch, int Z, long long HW,
                                  cudaStream_t st) {
  const unsigned g = grid_for((long long)N * Ch * Z * HW);
  if (dt == 0)
    batch_to_depth_kernel<0><<<g, 256, 0, st>>>(static_cast<const float*>(src), static_cast<float*>(dst), N, Ch, Z, HW);
  else
    batch_to_depth_kernel<1><<<g, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(src),
                                                 static_cast<__nv_bfloat16*>(dst), N, Ch, Z, HW);
  return cudaGetLastError();
}

cudaError_t launch_depth_scatter_add(int dt, const void* src, float* acc, int N, int Ch, int D, long long HW, int Z,
                                     int sd, int pd, int t, int dd, cudaStream_t st) {
  const unsigned g = grid_for((long long)N * Z * Ch * HW);
  if (dt == 0)
    depth_scatter_add_kernel<0><<<g, 256, 0, st>>>(static_cast<const float*>(src), acc, N, Ch, D, HW, Z, sd, pd, t, dd);
  else
    depth_scatter_add_kernel<1><<<g, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(src), acc, N, Ch, D, HW, Z, sd, pd,
                                                    t, dd);
  return cudaGetLastError();
}

cudaError_t launch_convert(int dt, const float* acc, void* dst, long long total, cudaStream_t st) {
  const unsigned g = grid_for(total);
  if (dt == 0)
    convert_kernel<0><<<g, 256, 0, st>>>(acc, static_cast<float*>(dst), total);
  else
    convert_kernel<1><<<g, 256, 0, st>>>(acc, static_cast<__nv_bfloat16*>(dst), total);
  return cudaGetLastError();
}

cudaError_t launch_filter_tap(int dt, const void* src, void* dst, long long KC, int T, int RS, int t, int to_slice,
                              cudaStream_t st) {
  const unsigned g = grid_for(KC * RS);
  if (dt == 0)
    filter_tap_kernel<0><<<g, 256, 0, st>>>(static_cast<const float*>(src), static_cast<float*>(dst), KC, T, RS, t,
                                             to_slice);
  else
    filter_tap_kernel<1><<<g, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(src), static_cast<__nv_bfloat16*>(dst), KC,
                                             T, RS, t, to_slice);
  return cudaGetLastError();
}

}  // namespace cg3

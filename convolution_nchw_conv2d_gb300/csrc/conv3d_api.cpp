// conv3d_api.cpp -- the 3-D (NCDHW) entry points of include/conv2d_gb300.h, built on the 2-D ones.
//
// A depth tap t of the filter reads input depth d = z*stride_d - pad_d + t*dil_d for output depth
// z, so each op is a sum over depth taps of 2-D operations on batches of depth slices:
//   forward          y[n,:,z]  = sum_t conv2d_fwd(x[n,:,d(z,t)], w[:,:,t])
//   backward-data    dx[n,:,d] = sum over (t, z) with d(z,t) = d of conv2d_bwd_data(dy[n,:,z], w[:,:,t])
//   backward-filter  dw[:,:,t] = conv2d_bwd_filter(x[n,:,d(z,t)], dy[n,:,z]) over all (n, z)
// Per depth tap, the slices d(z, t) of every image are gathered into a batch of N*Z images
// (zero where d leaves the tensor) and one 2-D call runs on it; the forward passes add onto
// their output (beta = 1 after the first), backward-data passes are added into an fp32 buffer
// placed at depth d(z, t), backward-filter passes write their filter slice.  The 2-D calls carry
// the height/width pads, strides, dilations and groups.  Workspace: the gathered batches, one
// filter slice, the fp32 buffer (backward-data), then the 2-D call's own workspace.
#include "conv2d_gb300.h"

#include <algorithm>
#include <cstdint>

#include <cuda_runtime.h>

namespace cg3 {
int count_launch(cudaError_t e, int kernels);
cudaError_t launch_depth_gather(int dt, const void* src, void* dst, int N, int Ch, int Dsrc, long long HW, int Zc,
                                int sd, int pd, int t, int dd, cudaStream_t st);
cudaError_t launch_batch_to_depth(int dt, const void* src, void* dst, int N, int Ch, int Z, long long HW,
                                  cudaStream_t st);
cudaError_t launch_depth_scatter_add(int dt, const void* src, float* acc, int N, int Ch, int D, long long HW, int Z,
                                     int sd, int pd, int t, int dd, cudaStream_t st);
cudaError_t launch_convert(int dt, const float* acc, void* dst, long long total, cudaStream_t st);
cudaError_t launch_filter_tap(int dt, const void* src, void* dst, long long KC, int T, int RS, int t, int to_slice,
                              cudaStream_t st);
}  // namespace cg3

namespace {

constexpr size_t kWsCap = 1000000000ull;  // the 2-D entry points' workspace cap

struct D3 {
  int N, C, D, H, W, K, T, R, S, pd, ph, pw, sd, sh, sw, dd, dh, dw, Z, P, Q;
  int groups, dt;
};

size_t al(size_t b) { return (b + 255) & ~size_t(255); }

int out3(int in, int pad, int k, int stride, int dil) {
  const int span = dil * (k - 1) + 1;
  const int num = in + 2 * pad - span;
  return num < 0 ? -1 : num / stride + 1;
}

int parse(const int* dims, int groups, int dtype, D3& d) {
  if (dims == nullptr) return CONV2D_ERR_NULLPTR;
  if (dtype != CONV2D_DTYPE_F32 && dtype != CONV2D_DTYPE_BF16) return CONV2D_ERR_DTYPE;
  d = D3{dims[0],  dims[1],  dims[2],  dims[3],  dims[4],  dims[5],  dims[6],  dims[7],  dims[8],  dims[9],  dims[10],
         dims[11], dims[12], dims[13], dims[14], dims[15], dims[16], dims[17], dims[18], dims[19], dims[20], groups,
         dtype};
  if (d.N < 1 || d.C < 1 || d.D < 1 || d.H < 1 || d.W < 1 || d.K < 1 || d.T < 1 || d.R < 1 || d.S < 1 || d.pd < 0 ||
      d.ph < 0 || d.pw < 0 || d.sd < 1 || d.sh < 1 || d.sw < 1 || d.dd < 1 || d.dh < 1 || d.dw < 1 || groups < 1 ||
      d.C % groups || d.K % groups)
    return CONV2D_ERR_BAD_DESC;
  if (out3(d.D, d.pd, d.T, d.sd, d.dd) < 1 || out3(d.H, d.ph, d.R, d.sh, d.dh) < 1 ||
      out3(d.W, d.pw, d.S, d.sw, d.dw) < 1)
    return CONV2D_ERR_SHAPE;
  if (d.Z != out3(d.D, d.pd, d.T, d.sd, d.dd) || d.P != out3(d.H, d.ph, d.R, d.sh, d.dh) ||
      d.Q != out3(d.W, d.pw, d.S, d.sw, d.dw))
    return CONV2D_ERR_SHAPE;
  const long long lim = 1ll << 31;
  if ((long long)d.N * d.Z * d.C * d.H * d.W >= lim || (long long)d.N * d.C * d.D * d.H * d.W >= lim ||
      (long long)d.N * d.K * d.Z * d.P * d.Q >= lim || (long long)d.K * (d.C / groups) * d.T * d.R * d.S >= lim)
    return CONV2D_ERR_TOO_LARGE;
  return CONV2D_OK;
}

// Workspace pieces of one op: the gathered source batch, the gathered second operand (dy for
// backward-data and -filter), the filter slice, the fp32 accumulator (backward-data), the 2-D
// call's workspace.
struct Ws {
  size_t src, src2, wt, acc, ws2, total;
};

int plan_ws(int op, const D3& d, Ws& w) {
  const size_t esz = d.dt == CONV2D_DTYPE_F32 ? 4 : 2;
  const size_t nx = (size_t)d.N * d.Z * d.C * d.H * d.W, ny = (size_t)d.N * d.Z * d.K * d.P * d.Q;
  const size_t nw = (size_t)d.K * (d.C / d.groups) * d.R * d.S;
  int rc = conv2d_workspace_size_ex(op, d.N * d.Z, d.C, d.H, d.W, d.K, d.R, d.S, d.ph, d.pw, d.sh, d.sw, d.P, d.Q,
                                    d.dh, d.dw, d.groups, d.dt, &w.ws2);
  if (rc) return rc;
  w.acc = 0;
  if (op == CONV2D_OP_FWD) {  // x batch, y batch, filter slice
    w.src = nx * esz;
    w.src2 = ny * esz;
    w.wt = nw * esz;
  } else if (op == CONV2D_OP_BWD_DATA) {  // dy batch, dx batch, filter slice, fp32 dx
    w.src = ny * esz;
    w.src2 = nx * esz;
    w.wt = nw * esz;
    w.acc = (size_t)d.N * d.C * d.D * d.H * d.W * sizeof(float);
  } else if (op == CONV2D_OP_BWD_FILTER) {  // x batch, dy batch, filter slice
    w.src = nx * esz;
    w.src2 = ny * esz;
    w.wt = nw * esz;
  } else {
    return CONV2D_ERR_BAD_OP;
  }
  w.total = al(w.src) + al(w.src2) + al(w.wt) + al(w.acc) + w.ws2;
  if (w.total > kWsCap) return CONV2D_ERR_UNSUPPORTED;
  return CONV2D_OK;
}

int check_ptrs3(const void* a, const void* b, const void* c, const void* ws, size_t wsb, const Ws& w, int dt) {
  if (!a || !b || !c) return CONV2D_ERR_NULLPTR;
  const uintptr_t m = dt == CONV2D_DTYPE_F32 ? 3 : 1;
  if (((uintptr_t)a & m) || ((uintptr_t)b & m) || ((uintptr_t)c & m)) return CONV2D_ERR_ALIGN;
  if (!ws) return CONV2D_ERR_NULLPTR;
  if ((uintptr_t)ws & 255) return CONV2D_ERR_ALIGN;
  if (wsb < w.total) return CONV2D_ERR_WORKSPACE;
  return CONV2D_OK;
}

uint8_t* at(void* base, size_t off) { return static_cast<uint8_t*>(base) + off; }

}  // namespace

extern "C" {

int conv3d_workspace_size(int op, const int* dims, int groups, int dtype, size_t* bytes) {
  if (!bytes) return CONV2D_ERR_NULLPTR;
  D3 d;
  int rc = parse(dims, groups, dtype, d);
  if (rc) return rc;
  Ws w;
  rc = plan_ws(op, d, w);
  if (rc) return rc;
  *bytes = w.total;
  return CONV2D_OK;
}

int conv3d_fwd(const int* dims, int groups, int dtype, const void* x, const void* w, void* y, void* workspace,
               size_t workspace_bytes, void* stream) {
  D3 d;
  int rc = parse(dims, groups, dtype, d);
  if (rc) return rc;
  Ws ws;
  rc = plan_ws(CONV2D_OP_FWD, d, ws);
  if (rc) return rc;
  rc = check_ptrs3(x, w, y, workspace, workspace_bytes, ws, dtype);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* xb = at(workspace, 0);
  void* yb = at(workspace, al(ws.src));
  void* wt = at(workspace, al(ws.src) + al(ws.src2));
  void* w2 = at(workspace, al(ws.src) + al(ws.src2) + al(ws.wt));
  const long long HW = (long long)d.H * d.W;
  const int Cg = d.C / groups;
  for (int t = 0; t < d.T; ++t) {
    rc = cg3::count_launch(cg3::launch_depth_gather(dtype, x, xb, d.N, d.C, d.D, HW, d.Z, d.sd, d.pd, t, d.dd, st), 1);
    if (rc) return rc;
    rc = cg3::count_launch(cg3::launch_filter_tap(dtype, w, wt, (long long)d.K * Cg, d.T, d.R * d.S, t, 1, st), 1);
    if (rc) return rc;
    rc = conv2d_fwd_ex(d.N * d.Z, d.C, d.H, d.W, d.K, d.R, d.S, d.ph, d.pw, d.sh, d.sw, d.P, d.Q, d.dh, d.dw, groups,
                       dtype, CONV2D_MODE_CROSS_CORRELATION, xb, wt, nullptr, t == 0 ? 0.f : 1.f, yb, w2, ws.ws2,
                       stream);
    if (rc) return rc;
  }
  return cg3::count_launch(cg3::launch_batch_to_depth(dtype, yb, y, d.N, d.K, d.Z, (long long)d.P * d.Q, st), 1);
}

int conv3d_bwd_data(const int* dims, int groups, int dtype, const void* dy, const void* w, void* dx, void* workspace,
                    size_t workspace_bytes, void* stream) {
  D3 d;
  int rc = parse(dims, groups, dtype, d);
  if (rc) return rc;
  Ws ws;
  rc = plan_ws(CONV2D_OP_BWD_DATA, d, ws);
  if (rc) return rc;
  rc = check_ptrs3(dy, w, dx, workspace, workspace_bytes, ws, dtype);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* dyb = at(workspace, 0);
  void* dxb = at(workspace, al(ws.src));
  void* wt = at(workspace, al(ws.src) + al(ws.src2));
  float* acc = reinterpret_cast<float*>(at(workspace, al(ws.src) + al(ws.src2) + al(ws.wt)));
  void* w2 = at(workspace, al(ws.src) + al(ws.src2) + al(ws.wt) + al(ws.acc));
  const long long HW = (long long)d.H * d.W;
  const int Cg = d.C / groups;
  // dy as a batch of N*Z images (one reshuffle for all taps); dx accumulated in fp32
  rc = cg3::count_launch(
      cg3::launch_depth_gather(dtype, dy, dyb, d.N, d.K, d.Z, (long long)d.P * d.Q, d.Z, 1, 0, 0, 1, st), 1);
  if (rc) return rc;
  if (cudaMemsetAsync(acc, 0, ws.acc, st) != cudaSuccess) return CONV2D_ERR_LAUNCH;
  for (int t = 0; t < d.T; ++t) {
    rc = cg3::count_launch(cg3::launch_filter_tap(dtype, w, wt, (long long)d.K * Cg, d.T, d.R * d.S, t, 1, st), 1);
    if (rc) return rc;
    rc = conv2d_bwd_data_ex(d.N * d.Z, d.C, d.H, d.W, d.K, d.R, d.S, d.ph, d.pw, d.sh, d.sw, d.P, d.Q, d.dh, d.dw,
                            groups, dtype, CONV2D_MODE_CROSS_CORRELATION, dyb, wt, nullptr, 0.f, dxb, w2, ws.ws2,
                            stream);
    if (rc) return rc;
    rc = cg3::count_launch(
        cg3::launch_depth_scatter_add(dtype, dxb, acc, d.N, d.C, d.D, HW, d.Z, d.sd, d.pd, t, d.dd, st), 1);
    if (rc) return rc;
  }
  return cg3::count_launch(cg3::launch_convert(dtype, acc, dx, (long long)d.N * d.C * d.D * HW, st), 1);
}

int conv3d_bwd_filter(const int* dims, int groups, int dtype, const void* x, const void* dy, void* dw, void* workspace,
                      size_t workspace_bytes, void* stream) {
  D3 d;
  int rc = parse(dims, groups, dtype, d);
  if (rc) return rc;
  Ws ws;
  rc = plan_ws(CONV2D_OP_BWD_FILTER, d, ws);
  if (rc) return rc;
  rc = check_ptrs3(x, dy, dw, workspace, workspace_bytes, ws, dtype);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* xb = at(workspace, 0);
  void* dyb = at(workspace, al(ws.src));
  void* wt = at(workspace, al(ws.src) + al(ws.src2));
  void* w2 = at(workspace, al(ws.src) + al(ws.src2) + al(ws.wt));
  const long long HW = (long long)d.H * d.W;
  const int Cg = d.C / groups;
  rc = cg3::count_launch(
      cg3::launch_depth_gather(dtype, dy, dyb, d.N, d.K, d.Z, (long long)d.P * d.Q, d.Z, 1, 0, 0, 1, st), 1);
  if (rc) return rc;
  for (int t = 0; t < d.T; ++t) {
    rc = cg3::count_launch(cg3::launch_depth_gather(dtype, x, xb, d.N, d.C, d.D, HW, d.Z, d.sd, d.pd, t, d.dd, st), 1);
    if (rc) return rc;
    rc = conv2d_bwd_filter_ex(d.N * d.Z, d.C, d.H, d.W, d.K, d.R, d.S, d.ph, d.pw, d.sh, d.sw, d.P, d.Q, d.dh, d.dw,
                              groups, dtype, CONV2D_MODE_CROSS_CORRELATION, xb, dyb, 0.f, wt, nullptr, nullptr, w2,
                              ws.ws2, stream);
    if (rc) return rc;
    rc = cg3::count_launch(cg3::launch_filter_tap(dtype, wt, dw, (long long)d.K * Cg, d.T, d.R * d.S, t, 0, st), 1);
    if (rc) return rc;
  }
  return CONV2D_OK;
}

}  // extern "C"

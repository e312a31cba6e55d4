// conv2d_api.cpp -- the C ABI (include/conv2d_gb300.h): descriptor validation,
// planning of the implicit-GEMM launches, workspace sizing and launch on the
// caller's stream.  No device memory is allocated here; nothing throws.
#include "conv2d_gb300.h"

#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "conv_plan.h"

namespace cg3 {
cudaError_t launch_tap_gemm(const TapPlan& p, int dt, int grid, cudaStream_t st);
cudaError_t launch_pack_filter(const PackPlan& pp, int dt, cudaStream_t st);
cudaError_t launch_dw_fwd(const DwPlan& p, int dt, int num_sms, cudaStream_t st);
cudaError_t launch_dw_bwd_data(const DwPlan& p, int dt, int num_sms, cudaStream_t st);
cudaError_t launch_dw_bwd_filter(const DwPlan& p, int dt, int num_sms, cudaStream_t st);
size_t tap_gemm_smem_bytes(const TapPlan& p);
cudaError_t launch_wgrad(const WgradPlan& p, int dt, int grid, cudaStream_t st);
cudaError_t launch_wgrad_reduce(const ReducePlan& rp, int dt, int num_sms, cudaStream_t st);
cudaError_t launch_chan_sum(const ChanSumPlan& a, const ChanSumPlan& b, int dt, cudaStream_t st);
cudaError_t launch_space_to_depth(const S2dPlan& sp, int dt, int num_sms, cudaStream_t st);
size_t wgrad_smem_bytes(const WgradPlan& p, int dt);
cudaError_t launch_wgrad_mn(const WgradMnPlan& p, int grid, cudaStream_t st);
cudaError_t launch_nhwc_pack(const NhwcPackPlan& a, const NhwcPackPlan& b, int dt, int num_sms, cudaStream_t st);
cudaError_t launch_tap_packs(const NhwcPackPlan& px, const PackPlan& pp, int dt, int num_sms, cudaStream_t st);
cudaError_t launch_wgrad_reduce_t(const ReduceTPlan& rp, int dt, int num_sms, cudaStream_t st);
size_t wgrad_mn_smem_bytes(const WgradMnPlan& p);
int tap_gemm_take_error();
int wgrad_take_error();
int wgrad_mn_take_error();
cudaError_t launch_c2i(const C2iPlan& p, int num_sms, cudaStream_t st);
size_t c2i_smem_bytes(const C2iPlan& p);
int c2i_take_error();
size_t noalloc_scratch_capacity();
cudaError_t noalloc_scratch_ptr(void** ptr);
}  // namespace cg3

using namespace cg3;

namespace {

constexpr size_t kWorkspaceCap = 1000000000ull;  // 1e9 bytes
constexpr int kMaxTapPasses = 16;                // tap passes of one forward / backward-data call
constexpr int kDefaultSMs = 152;                  // used when no device can be queried
constexpr size_t kDefaultSmemOptin = 232448;      // 227 KB

struct Desc {
  int N, C, H, W, K, R, S, ph, pw, sh, sw, P, Q, dt;
  int dh = 1, dw = 1;  // dilation: filter tap (r, s) sits at (r*dh, s*dw) in the window
  int g = 1;           // groups this per-group descriptor belongs to: the tensors hold g*C
                       // input and g*K output channels (image strides), the filter K x C
  int xg = 0;          // x image stride in units of C*H*W when not g (stride-phase planes)
};

int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }
int ceil_div_i(int a, int b) { return -floor_div(-a, b); }
int round_up(int a, int b) { return (a + b - 1) / b * b; }

int out_dim(int in, int pad, int k, int stride) {
  const int num = in + 2 * pad - k;
  if (num < 0) return 0;
  return num / stride + 1;
}

int validate(const Desc& d) {
  if (d.N <= 0 || d.C <= 0 || d.H <= 0 || d.W <= 0 || d.K <= 0 || d.R <= 0 || d.S <= 0 || d.ph < 0 ||
      d.pw < 0 || d.sh < 1 || d.sw < 1)
    return CONV2D_ERR_BAD_DESC;
  if (d.dt != CONV2D_DTYPE_F32 && d.dt != CONV2D_DTYPE_BF16) return CONV2D_ERR_DTYPE;
  // Overflow-safe: the sums below are bounded by 2^31 + 2^31.
  if (d.dh < 1 || d.dw < 1) return CONV2D_ERR_BAD_DESC;
  // extent of the dilated filter (overflow-safe: R, S, dh, dw are positive ints)
  const long long Re = (long long)d.dh * (d.R - 1) + 1, Se = (long long)d.dw * (d.S - 1) + 1;
  if (Re > INT_MAX || Se > INT_MAX) return CONV2D_ERR_BAD_DESC;
  const long long P = out_dim(d.H, d.ph, (int)Re, d.sh), Q = out_dim(d.W, d.pw, (int)Se, d.sw);
  if (P < 1 || Q < 1 || d.P != P || d.Q != Q) return CONV2D_ERR_SHAPE;
  const long long lim = (1ll << 31);
  if ((long long)d.N * d.C * d.H * d.W >= lim || (long long)d.N * d.K * d.P * d.Q >= lim ||
      (long long)d.K * d.C * d.R * d.S >= lim)
    return CONV2D_ERR_TOO_LARGE;
  // forward / backward-data run at most kMaxTapPasses passes of at most kMaxTaps taps;
  // backward-filter plans refuse more than kMaxTaps taps per stride phase themselves
  if ((long long)d.R * d.S > (long long)kMaxTapPasses * kMaxTaps || (long long)d.sh * d.sw > kMaxPlanes)
    return CONV2D_ERR_UNSUPPORTED;
  return CONV2D_OK;
}

// Per-group descriptor of a grouped problem (C and K are the totals; the filter is
// K x C/groups x R x S): C/groups input and K/groups output channels per group.
int group_desc(const Desc& d, int groups, Desc& dg) {
  if (groups < 1 || d.C % groups != 0 || d.K % groups != 0) return CONV2D_ERR_BAD_DESC;
  dg = d;
  dg.C = d.C / groups;
  dg.K = d.K / groups;
  dg.g = groups;
  return CONV2D_OK;
}

const uint8_t* byte_ptr(const void* p) { return static_cast<const uint8_t*>(p); }

// Depthwise layers (groups > 1 with one input channel per group) run the direct kernels of
// conv_depthwise.cu (DwPlan) instead of one tap-GEMM pass per group.
bool is_depthwise(const Desc& dg) { return dg.g > 1 && dg.C == 1; }
// Grouped layers (other than depthwise) whose forward and backward-data run as one pass over the
// whole tensors with a block-diagonally packed filter (run_tap); fp32 backward-data over 8 or
// fewer channels in all keeps the few-channel kernel per group.
bool blockdiag_groups(int op, const Desc& whole, int groups) {
  return groups >= 2 && (op == CONV2D_OP_FWD || whole.C > 8 || whole.dt != CONV2D_DTYPE_F32);
}

// The depthwise plan of a whole grouped problem (d: the totals; dg: its per-group descriptor);
// pointers, bias, beta and mode are set by the caller.  The filter gradient's splits are ranges
// of images, enough (K * splits blocks) for about eight blocks per SM.
DwPlan dw_plan(const Desc& d, const Desc& dg, int sms) {
  DwPlan p;
  std::memset(&p, 0, sizeof(p));
  p.N = d.N; p.C = d.C; p.H = d.H; p.W = d.W; p.K = d.K; p.R = d.R; p.S = d.S; p.P = d.P; p.Q = d.Q;
  p.ph = d.ph; p.pw = d.pw; p.sh = d.sh; p.sw = d.sw; p.dh = d.dh; p.dw = d.dw;
  p.M = dg.K;
  const int want = std::max(1, (8 * sms + d.K - 1) / d.K);
  p.n_per_split = std::max(1, (d.N + want - 1) / want);
  p.nsplit = (d.N + p.n_per_split - 1) / p.n_per_split;
  return p;
}

size_t dw_partial_bytes(const DwPlan& p) { return (size_t)p.nsplit * p.K * p.R * p.S * sizeof(float); }

struct DevInfo {
  int sms = kDefaultSMs;
  size_t smem_optin = kDefaultSmemOptin;
  bool ok = false;  // an sm_100-family device is current
};

std::mutex g_dev_mu;
std::vector<DevInfo> g_dev_cache;
std::vector<char> g_dev_known;

DevInfo device_info() {
  DevInfo di;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return di;
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if ((size_t)dev < g_dev_known.size() && g_dev_known[dev]) return g_dev_cache[dev];
  int major = 0, sms = 0, smem = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess) {
    di.sms = sms;
    di.smem_optin = (size_t)smem;
    di.ok = (major == 10);
  } else {
    cudaGetLastError();
  }
  if ((size_t)dev >= g_dev_known.size()) {
    g_dev_known.resize(dev + 1, 0);
    g_dev_cache.resize(dev + 1);
  }
  g_dev_cache[dev] = di;
  g_dev_known[dev] = 1;
  return di;
}

// A 1x1 filter with unit stride and no padding sees each image as one row of H*W
// pixels; planning it that way makes every row of the linear space contiguous.
Desc flatten_pointwise(Desc d) {
  // (P == H and Q == W for every caller descriptor of such a filter; a stride-phase problem
  // may carry a smaller output and is left as it is)
  if (d.R == 1 && d.S == 1 && d.ph == 0 && d.pw == 0 && d.sh == 1 && d.sw == 1 && d.P == d.H && d.Q == d.W) {
    d.W = d.H * d.W;
    d.H = 1;
    d.Q = d.W;
    d.P = 1;
  }
  return d;
}

// ------------------------------------------------------------------ tap plans
struct TapBuild {
  TapPlan p;
  PackPlan pp;
  size_t pack_bytes;
  int grid;
  NhwcPackPlan px;        // channel-chunk pack of the source planes (when p.a_tma)
  size_t src_pack_bytes;  // its size: planes * chunks * positions * 16 bytes
};

bool setup_pack_tiles(NhwcPackPlan& q, int esz);
bool encode_mn_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint32_t* box);
bool encode_tap_src_map(TapPlan& p, const void* base, int nchunk, int npl, int dt);

// MMA operand offsets of every tap within a pipeline stage, in 16-byte units, once the tile
// shape (NCH channel chunks of `rows` rows per plane, NT filter rows per chunk) is fixed.  A
// stage holds, per source plane, NCH chunk blocks of `rows` position rows, and per tap of the
// phase NCH chunk blocks of NT filter rows.  In tap-pair mode (NCH == 1) the even tap of each
// pair also carries the row distance to the odd tap in bits 16..29, the field the descriptor
// reads as its K-direction (leading byte) offset, so that one K = 2-chunk MMA covers both.
void fill_tap_offsets(TapPlan& p, int NCH) {
  for (int ph = 0; ph < p.nph; ++ph)
    for (int i = 0; i < p.ph_ntaps[ph]; ++i) {
      const int t = p.ph_tap_begin[ph] + i;
      const int spl = p.plane_per_phase ? 0 : p.tap_plane[t];  // plane within the stage
      const int oa = spl * NCH * p.rows + p.tap_off[t];
      if (NCH >= 2) {
        p.tap_a[t] = oa;
        p.tap_b[t] = i * NCH * p.NT;
      } else if ((i & 1) == 0) {
        const int ob = (p.plane_per_phase ? 0 : p.tap_plane[t + 1]) * p.rows + p.tap_off[t + 1];
        p.tap_a[t] = (int)((uint32_t)oa | ((uint32_t)(ob - oa) << 16));
        p.tap_b[t] = i * p.NT;
      } else {
        p.tap_a[t] = 0;
        p.tap_b[t] = 0;
      }
    }
}

// Chooses MH, NT, CB, ACCB and the stage count for a TapPlan whose geometry (linear
// space, planes, phases, taps) is already filled in.  Returns false if nothing fits.
bool choose_tap_tiles(TapPlan& p, int max_off, int dt, const DevInfo& di, bool pair_taps, bool a_tma) {
  const int CHUNK = dt == 0 ? 4 : 8;
  const size_t budget = di.smem_optin - 2048;
  int nt_cands[2];
  int nnt = 0;
  if (p.Cd <= 256) {
    nt_cands[nnt++] = round_up(p.Cd, 16);
  } else {
    nt_cands[nnt++] = 256;
    nt_cands[nnt++] = 128;
  }
  int cb_cands[4];
  int ncand = 0;
  if (pair_taps) {
    cb_cands[ncand++] = CHUNK;
  } else {
    const int cmax = round_up(p.Cs, 2 * CHUNK);
    for (int cb : {16 * CHUNK, 8 * CHUNK, 4 * CHUNK, 2 * CHUNK})
      if (cb <= cmax || cb == 2 * CHUNK) cb_cands[ncand++] = cb;
  }
  for (int ni = 0; ni < nnt; ++ni) {
    const int NT = nt_cands[ni];
    const int n_ntiles = (p.Cd + NT - 1) / NT;
    for (int mh = 2; mh >= 1; --mh) {
      const long long mtiles = (p.Mtot + 128ll * mh - 1) / (128ll * mh);
      // Small problems: prefer more, smaller tiles so that every SM gets work.
      if (mh == 2 && mtiles * n_ntiles * p.nph < di.sms) continue;
      // Keep two accumulator buffers in TMEM (the epilogue of one tile overlaps the
      // mainloop of the next): two 128-row halves only when 4*NT columns fit.
      if (mh == 2 && 4 * NT > 512) continue;
      for (int ci = 0; ci < ncand; ++ci) {
        const int CB = cb_cands[ci];
        const int NCH = CB / CHUNK;
        int rows = round_up(128 * mh + max_off + (pair_taps ? 1 : 0), 8);
        // tensor-copied rows: equal boxes of at most 128 rows (256 8-byte elements), a multiple
        // of 8 rows each; the box count that pads the rows least
        int nbox = 1, box = rows;
        if (a_tma) {
          const int n0 = (rows + 127) / 128;
          box = 1 << 30;
          for (int nb = n0; nb < n0 + 4; ++nb) {
            const int bx = round_up((rows + nb - 1) / nb, 8);
            if (nb * bx < nbox * box) {
              nbox = nb;
              box = bx;
            }
          }
        }
        rows = nbox * box;
        if (a_tma && 2 * (p.Mtot + rows) >= (1ll << 31)) return false;  // 32-bit copy coordinates
        const long long a_bytes = (long long)(p.plane_per_phase ? 1 : p.npl) * NCH * rows * 16;
        const long long b_bytes = (long long)p.max_taps_ph * NCH * NT * 16;
        const long long fixed = 8 * (3 * 4 + 6) + 24 + 4 * 4 + 1024;
        const long long per = a_bytes + b_bytes;
        long long stages = ((long long)budget - fixed) / per;
        if (stages < 2) continue;
        if (stages > 4) stages = 4;
        if (b_bytes + (a_tma ? a_bytes : 0) >= (1 << 20)) continue;  // mbarrier transaction-count limit
        p.NT = NT;
        p.n_ntiles = n_ntiles;
        p.MH = mh;
        p.CB = CB;
        p.rows = rows;
        p.a_tma = a_tma ? 1 : 0;
        p.a_box = box;
        p.a_nbox = nbox;
        // One copy per stage for stages of several planes (stride-phase planes of the forward
        // op), where it replaced 8 copies and measured faster; single-plane stages keep the
        // copies of a_box rows (one copy measured no faster there).  A box is at most 256 in
        // every dimension.
        p.a_one = a_tma && !p.plane_per_phase && p.npl > 1 && rows <= 256 ? 1 : 0;
        p.a_stage_bytes = (int)a_bytes;
        p.b_stage_bytes = (int)b_bytes;
        p.stages = (int)stages;
        p.ACCB = (2 * mh * NT <= 512) ? 2 : 1;
        p.tmem_cols = 32;
        while (p.tmem_cols < p.ACCB * mh * NT) p.tmem_cols <<= 1;
        p.nkb = (p.Cs + CB - 1) / CB;
        p.n_mtiles = (int)mtiles;
        p.total_tiles = (long long)p.nph * p.n_mtiles * p.n_ntiles;
        if (tap_gemm_smem_bytes(p) <= di.smem_optin) {
          fill_tap_offsets(p, NCH);
          return true;
        }
      }
    }
  }
  return false;
}

// The channel-chunk pack of a tap plan's source planes: plane pl at linear position
// L = n*EL*WL + e*WL + f holds the source pixel (e*pl_step_h + pl_off_h[pl], f*pl_step_w +
// pl_off_w[pl]) of image n, zero outside the tensor -- the pixel the producers' direct loads
// read for staged row L.  The destination is set once the workspace is laid out.
void fill_src_pack(TapBuild& b, int dt) {
  const TapPlan& p = b.p;
  NhwcPackPlan& q = b.px;
  std::memset(&q, 0, sizeof(q));
  const int CHUNK = dt == 0 ? 4 : 8;
  q.src = p.src;
  q.src_nstride = p.src_nstride;
  q.N = p.N;
  q.C = p.Cs;
  q.H = p.Hs;
  q.W = p.Ws;
  q.nchunk = (p.Cs + CHUNK - 1) / CHUNK;
  q.EX = p.EL;
  q.WL = p.WL;
  q.fd_WL = make_fastdiv((uint32_t)p.WL);
  q.npl = p.npl;
  q.step_h = p.pl_step_h;
  q.step_w = p.pl_step_w;
  for (int pl = 0; pl < p.npl; ++pl) {
    q.off_h[pl] = p.pl_off_h[pl];
    q.off_w[pl] = p.pl_off_w[pl];
  }
  b.src_pack_bytes = (size_t)q.npl * q.nchunk * (size_t)p.Mtot * 16;
}

// Packed-source staging is planned when the caller allows the workspace for it, the pack has a
// work-unit tiling (fill_src_pack, then setup_pack_tiles), and the copy pays: bf16 sources, and
// fp32 sources of one channel chunk (the direct loads then fill a quarter of each staged row
// with 3 or fewer channels).  For fp32 sources of several chunks the extra pass over the
// 4-byte tensor costs more than the staging it saves (measured on the 3x3, strided and 1x1
// layers: the direct producers keep up with the MMAs there).
bool packed_src_ok(TapBuild& b, int dt) {
  if (dt == 0 && b.p.Cs > 4) return false;
  fill_src_pack(b, dt);
  return setup_pack_tiles(b.px, dt == 0 ? 4 : 2);
}

void fill_pack(TapBuild& b, const Desc& d, const void* w, void* wpack, int transpose,
               const std::vector<int>& tr, const std::vector<int>& ts) {
  PackPlan& pp = b.pp;
  std::memset(&pp, 0, sizeof(pp));
  pp.w = w;
  pp.wpack = wpack;
  pp.K = d.K;
  pp.C = d.C;
  pp.R = d.R;
  pp.S = d.S;
  pp.transpose = transpose;
  pp.Cd = b.p.Cd;
  pp.Cs = b.p.Cs;
  pp.n_ntiles = b.p.n_ntiles;
  pp.nkb = b.p.nkb;
  pp.ntaps_total = b.p.ntaps_total;
  pp.NT = b.p.NT;
  pp.CB = b.p.CB;
  for (int t = 0; t < b.p.ntaps_total; ++t) {
    pp.tap_r[t] = tr[t];
    pp.tap_s[t] = ts[t];
  }
  const int CHUNK = d.dt == 0 ? 4 : 8;
  b.pack_bytes = (size_t)b.p.n_ntiles * b.p.nkb * b.p.ntaps_total * (b.p.CB / CHUNK) * b.p.NT * 16;
}

// Sort one phase's taps by staged address and, when taps are paired, pad to an even
// count with a zero-weight tap (weight coordinates -1) placed at the last real tap.
void order_phase_taps(std::vector<int>& pl, std::vector<int>& off, std::vector<int>& tr,
                      std::vector<int>& ts, int begin, int rows_hint, bool pair) {
  const int n = (int)pl.size() - begin;
  std::vector<int> idx(n);
  for (int i = 0; i < n; ++i) idx[i] = begin + i;
  std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) {
    const long long ka = (long long)pl[a] * rows_hint + off[a];
    const long long kb = (long long)pl[b] * rows_hint + off[b];
    return ka < kb;
  });
  std::vector<int> npl(n), noff(n), ntr(n), nts(n);
  for (int i = 0; i < n; ++i) {
    npl[i] = pl[idx[i]];
    noff[i] = off[idx[i]];
    ntr[i] = tr[idx[i]];
    nts[i] = ts[idx[i]];
  }
  for (int i = 0; i < n; ++i) {
    pl[begin + i] = npl[i];
    off[begin + i] = noff[i];
    tr[begin + i] = ntr[i];
    ts[begin + i] = nts[i];
  }
  if (pair && (n & 1)) {
    pl.push_back(pl.back());
    off.push_back(off.back());
    tr.push_back(-1);
    ts.push_back(-1);
  }
}

// Taps u = r*S + s in [u_lo, u_hi) only (the whole filter by default).  A partial tap set
// moves the staged window down by its smallest tap row (plane offsets up, tap offsets
// down by the same rows), so that the window holds no rows that none of its taps reads.
int build_fwd_impl(const Desc& d0, const void* x, const void* w, void* y, void* ws, const DevInfo& di,
                   TapBuild& b, int u_lo, int u_hi, bool packed_src, bool pair) {
  const Desc d = flatten_pointwise(d0);
  TapPlan& p = b.p;
  std::memset(&p, 0, sizeof(p));
  b.src_pack_bytes = 0;
  p.src = x;
  p.dst = y;
  p.N = d.N;
  p.Cs = d.C;
  p.Hs = d.H;
  p.Ws = d.W;
  p.Cd = d.K;
  p.Hd = d.P;
  p.Wd = d.Q;
  p.src_nstride = (long long)d.g * d.C * d.H * d.W;
  p.dst_nstride = (long long)d.g * d.K * d.P * d.Q;
  const int mh = (d.dh * (d.R - 1)) / d.sh, mw = (d.dw * (d.S - 1)) / d.sw;
  const int CHUNK = d.dt == 0 ? 4 : 8;
  p.WL = d.Q + mw;
  p.EL = d.P + mh;
  p.Mtot = (long long)d.N * p.EL * p.WL;
  if (p.Mtot >= (1ll << 31)) return CONV2D_ERR_TOO_LARGE;
  p.fd_img = make_fastdiv((uint32_t)(p.EL * p.WL));
  p.fd_WL = make_fastdiv((uint32_t)p.WL);
  p.npl = d.sh * d.sw;
  p.pl_step_h = d.sh;
  p.pl_step_w = d.sw;
  for (int a = 0; a < d.sh; ++a)
    for (int bb = 0; bb < d.sw; ++bb) {
      p.pl_off_h[a * d.sw + bb] = a - d.ph;
      p.pl_off_w[a * d.sw + bb] = bb - d.pw;
    }
  p.nph = 1;
  p.ph_step_h = 1;
  p.ph_step_w = 1;
  std::vector<int> tpl, toff, tr, ts;
  int min_row = 1 << 30;
  for (int r = 0; r < d.R; ++r)
    for (int s = 0; s < d.S; ++s) {
      if (r * d.S + s < u_lo || r * d.S + s >= u_hi) continue;
      const int re = r * d.dh, se = s * d.dw;  // the tap's place in the dilated window
      tpl.push_back((re % d.sh) * d.sw + (se % d.sw));
      toff.push_back((re / d.sh) * p.WL + se / d.sw);
      tr.push_back(r);
      ts.push_back(s);
      min_row = std::min(min_row, re / d.sh);
    }
  if (tpl.empty()) return CONV2D_ERR_BAD_DESC;
  int max_off = 0;
  for (int& o : toff) {
    o -= min_row * p.WL;
    max_off = std::max(max_off, o);
  }
  for (int pl = 0; pl < p.npl; ++pl) p.pl_off_h[pl] += min_row * d.sh;
  order_phase_taps(tpl, toff, tr, ts, 0, 1 << 20, pair);
  p.ntaps_total = (int)tpl.size();
  if (p.ntaps_total > kMaxTaps) return CONV2D_ERR_UNSUPPORTED;
  p.ph_tap_begin[0] = 0;
  p.ph_ntaps[0] = p.ntaps_total;
  p.max_taps_ph = p.ntaps_total;
  for (int t = 0; t < p.ntaps_total; ++t) {
    p.tap_plane[t] = tpl[t];
    p.tap_off[t] = toff[t];
  }
  const bool a_tma = packed_src && packed_src_ok(b, d.dt);
  if (!choose_tap_tiles(p, max_off, d.dt, di, pair, a_tma) && !(a_tma && choose_tap_tiles(p, max_off, d.dt, di, pair, false)))
    return CONV2D_ERR_UNSUPPORTED;
  if (!p.a_tma) b.src_pack_bytes = 0;
  p.wpack = ws;
  fill_pack(b, d, w, ws, 0, tr, ts);
  if (b.pack_bytes / 16 >= (size_t(1) << 31)) return CONV2D_ERR_TOO_LARGE;  // 32-bit chunk indices
  b.grid = (int)std::min<long long>(p.total_tiles, di.sms);
  return CONV2D_OK;
}

// Taps u = r*S + s in [u_lo, u_hi) only, with the staged window moved down by the
// smallest tap row as in build_fwd.
int build_bwd_data_impl(const Desc& d0, const void* dy, const void* w, void* dx, void* ws, const DevInfo& di,
                        TapBuild& b, int u_lo, int u_hi, bool packed_src, bool pair) {
  const Desc d = flatten_pointwise(d0);
  TapPlan& p = b.p;
  std::memset(&p, 0, sizeof(p));
  b.src_pack_bytes = 0;
  p.src = dy;
  p.dst = dx;
  p.N = d.N;
  p.Cs = d.K;
  p.Hs = d.P;
  p.Ws = d.Q;
  p.Cd = d.C;
  p.Hd = d.H;
  p.Wd = d.W;
  p.src_nstride = (long long)d.g * d.K * d.P * d.Q;
  p.dst_nstride = (long long)d.g * d.C * d.H * d.W;
  // Per output phase a (rows with (h + pad_h) mod stride_h == a): the taps r with
  // r*dh = a (mod stride_h), at t_r = (r*dh - a) / stride_h; output row h = sh*u + a - pad_h
  // reads dy row p = u - t_r.  Th[a] = 1 + the largest t_r (0: no tap reaches the phase).
  // Same for columns.
  auto phase_dims = [](int H, int pad, int R, int dil, int st, std::vector<int>& T, std::vector<int>& ulo,
                       std::vector<int>& U, std::vector<std::vector<int>>& taps) {
    T.assign(st, 0);
    ulo.assign(st, 0);
    U.assign(st, 0);
    taps.assign(st, {});
    for (int a = 0; a < st; ++a) {
      for (int r = 0; r < R; ++r)
        if ((r * dil) % st == a) {
          taps[a].push_back(r);
          T[a] = std::max(T[a], (r * dil - a) / st + 1);
        }
      ulo[a] = ceil_div_i(pad - a, st);
      const int uhi = floor_div(H - 1 + pad - a, st);
      U[a] = std::max(0, uhi - ulo[a] + 1);
    }
  };
  std::vector<int> Th, uloh, Uh, Tw, ulow, Uw;
  std::vector<std::vector<int>> tapsh, tapsw;
  phase_dims(d.H, d.ph, d.R, d.dh, d.sh, Th, uloh, Uh, tapsh);
  phase_dims(d.W, d.pw, d.S, d.dw, d.sw, Tw, ulow, Uw, tapsw);
  const int CHUNK = d.dt == 0 ? 4 : 8;
  // With the source packed for tensor copies (whole filter in one pass), every phase reads the
  // one packed dy plane from its own origin: phase (a, c) at linear (e, f) reads dy row
  // e + (Th[a]-1 - t_r) + dh_a and column f + (Tw[c]-1 - t_s) + dw_c with dh_a = ulo_a - (Th[a]-1),
  // dw_c likewise, i.e. the plane at linear position L + tap offset + dh_a*WL + dw_c.  The grid
  // (EL x WL per image) is large enough that every position a phase reads either lies in its
  // own image's rows or falls on zero rows / columns of the grid (a read before row 0 lands on
  // the previous image's last rows, which lie past P): EL >= U + T - 1, >= ulo + U and
  // >= P + T - 1 - ulo for every phase, likewise WL.  Each phase's linear space then spans its
  // own outputs, not the union of all phases' windows, so fewer position tiles, and the pack
  // writes dy once.
  if (packed_src && u_lo == 0 && u_hi >= d.R * d.S && d.sh * d.sw > 1) {
    int EL = std::max(1, d.P), WL = std::max(1, d.Q);
    for (int a = 0; a < d.sh; ++a) {
      EL = std::max(EL, Uh[a]);
      if (Th[a] > 0) EL = std::max({EL, Uh[a] + Th[a] - 1, Uh[a] + uloh[a], d.P + Th[a] - 1 - uloh[a]});
    }
    for (int c = 0; c < d.sw; ++c) {
      WL = std::max(WL, Uw[c]);
      if (Tw[c] > 0) WL = std::max({WL, Uw[c] + Tw[c] - 1, Uw[c] + ulow[c], d.Q + Tw[c] - 1 - ulow[c]});
    }
    TapPlan q = p;
    q.WL = WL;
    q.EL = EL;
    q.Mtot = (long long)d.N * EL * WL;
    if (q.Mtot < (1ll << 30)) {  // room for the phase shifts in the copies' 32-bit coordinates
      q.fd_img = make_fastdiv((uint32_t)(EL * WL));
      q.fd_WL = make_fastdiv((uint32_t)WL);
      q.npl = 1;
      q.nph = d.sh * d.sw;
      q.plane_per_phase = 1;
      q.pl_step_h = q.pl_step_w = 1;
      q.pl_off_h[0] = q.pl_off_w[0] = 0;
      q.ph_step_h = d.sh;
      q.ph_step_w = d.sw;
      std::vector<int> tpl, toff, tr, ts;
      int max_taps = 0, max_off = 0;
      for (int a = 0; a < d.sh; ++a)
        for (int c = 0; c < d.sw; ++c) {
          const int ph = a * d.sw + c;
          q.ph_shift[ph] = (uloh[a] - (std::max(Th[a], 1) - 1)) * WL + (ulow[c] - (std::max(Tw[c], 1) - 1));
          q.ph_off_h[ph] = d.sh * uloh[a] + a - d.ph;
          q.ph_off_w[ph] = d.sw * ulow[c] + c - d.pw;
          const int begin = (int)tpl.size();
          q.ph_tap_begin[ph] = begin;
          for (const int r : tapsh[a])
            for (const int s2 : tapsw[c]) {
              const int t = (r * d.dh - a) / d.sh, t2 = (s2 * d.dw - c) / d.sw;
              tpl.push_back(0);
              toff.push_back((Th[a] - 1 - t) * WL + (Tw[c] - 1 - t2));
              tr.push_back(r);
              ts.push_back(s2);
            }
          if ((int)tpl.size() > begin) order_phase_taps(tpl, toff, tr, ts, begin, 1 << 20, pair);
          q.ph_ntaps[ph] = (int)tpl.size() - begin;
          max_taps = std::max(max_taps, q.ph_ntaps[ph]);
        }
      for (const int o : toff) max_off = std::max(max_off, o);
      q.ntaps_total = (int)tpl.size();
      q.max_taps_ph = std::max(1, max_taps);
      if (q.ntaps_total > 0 && q.ntaps_total <= kMaxTaps) {
        for (int t = 0; t < q.ntaps_total; ++t) {
          q.tap_plane[t] = tpl[t];
          q.tap_off[t] = toff[t];
        }
        TapBuild bq = b;
        bq.p = q;
        if (packed_src_ok(bq, d.dt) && choose_tap_tiles(bq.p, max_off, d.dt, di, pair, true)) {
          bq.p.wpack = ws;
          fill_pack(bq, d, w, ws, 1, tr, ts);
          if (bq.pack_bytes / 16 < (size_t(1) << 31)) {
            bq.grid = (int)std::min<long long>(bq.p.total_tiles, di.sms);
            b = bq;
            return CONV2D_OK;
          }
        }
      }
    }
  }
  int T0h = 0, T0w = 0;
  for (int a = 0; a < d.sh; ++a)
    if (Th[a] > 0) T0h = std::max(T0h, Th[a] - 1 - uloh[a]);
  for (int c = 0; c < d.sw; ++c)
    if (Tw[c] > 0) T0w = std::max(T0w, Tw[c] - 1 - ulow[c]);
  int EL = 1, WL = 1;
  for (int a = 0; a < d.sh; ++a) {
    EL = std::max(EL, Uh[a]);
    if (Th[a] > 0) EL = std::max(EL, Uh[a] + uloh[a] + T0h);
  }
  for (int c = 0; c < d.sw; ++c) {
    WL = std::max(WL, Uw[c]);
    if (Tw[c] > 0) WL = std::max(WL, Uw[c] + ulow[c] + T0w);
  }
  p.WL = WL;
  p.EL = EL;
  p.Mtot = (long long)d.N * EL * WL;
  if (p.Mtot >= (1ll << 31)) return CONV2D_ERR_TOO_LARGE;
  p.fd_img = make_fastdiv((uint32_t)(EL * WL));
  p.fd_WL = make_fastdiv((uint32_t)WL);
  p.npl = 1;
  p.pl_step_h = 1;
  p.pl_step_w = 1;
  p.pl_off_h[0] = -T0h;
  p.pl_off_w[0] = -T0w;
  p.nph = d.sh * d.sw;
  p.ph_step_h = d.sh;
  p.ph_step_w = d.sw;
  std::vector<int> tpl, toff, tr, ts;
  int max_taps = 0, min_row = 1 << 30, n_real = 0;
  for (int a = 0; a < d.sh; ++a)
    for (int c = 0; c < d.sw; ++c)
      for (const int r : tapsh[a])
        for (const int s2 : tapsw[c])
          if (r * d.S + s2 >= u_lo && r * d.S + s2 < u_hi) {
            min_row = std::min(min_row, uloh[a] - (r * d.dh - a) / d.sh + T0h);
            ++n_real;
          }
  if (n_real == 0) {
    if (u_lo > 0 || u_hi < d.R * d.S) return CONV2D_ERR_BAD_DESC;
    min_row = 0;  // no tap reaches any output: the plan writes zeros
  }
  p.pl_off_h[0] += min_row;
  for (int a = 0; a < d.sh; ++a)
    for (int c = 0; c < d.sw; ++c) {
      const int ph = a * d.sw + c;
      p.ph_off_h[ph] = d.sh * uloh[a] + a - d.ph;
      p.ph_off_w[ph] = d.sw * ulow[c] + c - d.pw;
      const int begin = (int)tpl.size();
      p.ph_tap_begin[ph] = begin;
      for (const int r : tapsh[a])
        for (const int s2 : tapsw[c]) {
          if (r * d.S + s2 < u_lo || r * d.S + s2 >= u_hi) continue;
          const int t = (r * d.dh - a) / d.sh, t2 = (s2 * d.dw - c) / d.sw;
          const int roff = uloh[a] - t + T0h - min_row;
          const int coff = ulow[c] - t2 + T0w;
          tpl.push_back(0);
          toff.push_back(roff * WL + coff);
          tr.push_back(r);
          ts.push_back(s2);
        }
      if ((int)tpl.size() > begin) order_phase_taps(tpl, toff, tr, ts, begin, 1 << 20, pair);
      p.ph_ntaps[ph] = (int)tpl.size() - begin;
      max_taps = std::max(max_taps, p.ph_ntaps[ph]);
    }
  int max_off = 0;
  for (const int o : toff) max_off = std::max(max_off, o);
  p.ntaps_total = (int)tpl.size();
  if (p.ntaps_total > kMaxTaps) return CONV2D_ERR_UNSUPPORTED;
  p.max_taps_ph = std::max(1, max_taps);
  for (int t = 0; t < p.ntaps_total; ++t) {
    p.tap_plane[t] = tpl[t];
    p.tap_off[t] = toff[t];
  }
  const bool a_tma = packed_src && p.ntaps_total > 0 && packed_src_ok(b, d.dt);
  if (!choose_tap_tiles(p, max_off, d.dt, di, pair, a_tma) && !(a_tma && choose_tap_tiles(p, max_off, d.dt, di, pair, false)))
    return CONV2D_ERR_UNSUPPORTED;
  if (!p.a_tma) b.src_pack_bytes = 0;
  p.wpack = ws;
  fill_pack(b, d, w, ws, 1, tr, ts);
  if (p.ntaps_total == 0) b.pack_bytes = 0;
  if (b.pack_bytes / 16 >= (size_t(1) << 31)) return CONV2D_ERR_TOO_LARGE;  // 32-bit chunk indices
  b.grid = (int)std::min<long long>(p.total_tiles, di.sms);
  return CONV2D_OK;
}

// Tap-pair mode (one MMA of K = two 16-byte chunks covers one chunk of two taps) is natural
// when the source has at most one chunk of channels.  With more channels a stage normally holds
// two or more chunks of every tap of the phase; when that caps the tile's N below what the
// destination channels want, pair mode, whose stages hold one chunk (half the filter slice),
// is planned as well and kept if it reaches a wider N.
template <class Impl>
int build_tap_pass(Impl impl, int Cs, int Cd, int dt, TapBuild& b) {
  const int CHUNK = dt == 0 ? 4 : 8;
  const bool natural = Cs <= CHUNK;
  const int rc = impl(b, natural);
  if (natural || (rc != CONV2D_OK && rc != CONV2D_ERR_UNSUPPORTED)) return rc;
  if (rc == CONV2D_OK && b.p.NT >= std::min(256, round_up(Cd, 16))) return rc;
  TapBuild b2;
  const int rc2 = impl(b2, true);
  if (rc2 == CONV2D_OK && (rc != CONV2D_OK || b2.p.NT > b.p.NT)) {
    b = b2;
    return CONV2D_OK;
  }
  return rc;
}

int build_fwd(const Desc& d, const void* x, const void* w, void* y, void* ws, const DevInfo& di, TapBuild& b,
              int u_lo = 0, int u_hi = 1 << 30, bool packed_src = false) {
  return build_tap_pass(
      [&](TapBuild& bb, bool pair) { return build_fwd_impl(d, x, w, y, ws, di, bb, u_lo, u_hi, packed_src, pair); },
      d.C, d.K, d.dt, b);
}

int build_bwd_data(const Desc& d, const void* dy, const void* w, void* dx, void* ws, const DevInfo& di, TapBuild& b,
                   int u_lo = 0, int u_hi = 1 << 30, bool packed_src = false) {
  return build_tap_pass(
      [&](TapBuild& bb, bool pair) { return build_bwd_data_impl(d, dy, w, dx, ws, di, bb, u_lo, u_hi, packed_src, pair); },
      d.K, d.C, d.dt, b);
}

// ------------------------------------------------------------------ tensor maps
// cuTensorMapEncodeTiled, looked up once through the runtime (no link-time dependency on
// the driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess && f)
      fn = reinterpret_cast<EncodeTiledFn>(f);
    else
      cudaGetLastError();
  });
  return fn;
}

// x (N, C, H, W) as the 4-D tensor (w = W, h = H, c = C, n = N) with a box of one image row
// segment of WL pixels by 32 channels.  False if it cannot be encoded.
bool encode_x_map(CUtensorMap* m, const void* x, int dt, int N, int C, int H, int W, int WL, long long nstride) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const uint64_t esz = dt == 0 ? 4 : 2;
  const cuuint64_t dims[4] = {(cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)C, (cuuint64_t)N};
  const cuuint64_t strides[3] = {(cuuint64_t)W * esz, (cuuint64_t)H * W * esz, (cuuint64_t)nstride * esz};
  const cuuint32_t box[4] = {(cuuint32_t)WL, 1u, 32u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUresult r = fn(m, dt == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                        const_cast<void*>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// dy (N, K, P, Q) as the 4-D tensor (w = Q, k = K, e = P, n = N) with a box of one
// 16-byte chunk of positions by NK output channels.  False if it cannot be encoded.
bool encode_dy_map(CUtensorMap* m, const void* dy, int dt, int N, int K, int P, int Q, int NK, long long nstride) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const uint64_t esz = dt == 0 ? 4 : 2;
  const cuuint64_t dims[4] = {(cuuint64_t)Q, (cuuint64_t)K, (cuuint64_t)P, (cuuint64_t)N};
  const cuuint64_t strides[3] = {(cuuint64_t)P * Q * esz, (cuuint64_t)Q * esz, (cuuint64_t)nstride * esz};
  const cuuint32_t box[4] = {(cuuint32_t)(16 / esz), (cuuint32_t)NK, 1u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUresult r = fn(m, dt == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                        const_cast<void*>(dy), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// dy (N, K, P, Q) as the 5-D tensor (w mod CHUNK, k, w / CHUNK, e, n) with a box of one
// linear row of WL positions by NK output channels: shared-memory layout [chunk][k][CHUNK].
// False if it cannot be encoded.
bool encode_dy_row_map(CUtensorMap* m, const void* dy, int dt, int N, int K, int P, int Q, int NK, int WL,
                       long long nstride) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const uint64_t esz = dt == 0 ? 4 : 2;
  const uint64_t chunk = 16 / esz;
  const cuuint64_t dims[5] = {(cuuint64_t)chunk, (cuuint64_t)K, (cuuint64_t)(Q / chunk), (cuuint64_t)P,
                              (cuuint64_t)N};
  const cuuint64_t strides[4] = {(cuuint64_t)P * Q * esz, 16u, (cuuint64_t)Q * esz, (cuuint64_t)nstride * esz};
  const cuuint32_t box[5] = {(cuuint32_t)chunk, (cuuint32_t)NK, (cuuint32_t)(WL / chunk), 1u, 1u};
  const cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
  const CUresult r = fn(m, dt == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5,
                        const_cast<void*>(dy), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ wgrad plan
struct WgradBuild {
  WgradPlan p;
  ReducePlan rp;
  size_t partial_bytes;
  int grid;
};

int build_bwd_filter_impl(const Desc& d0, const void* x, const void* dy, void* dw, void* ws, const DevInfo& di,
                          WgradBuild& b, bool allow_tma, bool allow_rowshare) {
  const Desc d = flatten_pointwise(d0);
  WgradPlan& p = b.p;
  std::memset(&p, 0, sizeof(p));
  p.x = x;
  p.dy = dy;
  p.x_nstride = (long long)(d.xg ? d.xg : d.g) * d.C * d.H * d.W;
  p.dy_nstride = (long long)d.g * d.K * d.P * d.Q;
  p.partial = static_cast<float*>(ws);
  p.N = d.N;
  p.C = d.C;
  p.H = d.H;
  p.W = d.W;
  p.K = d.K;
  p.P = d.P;
  p.Q = d.Q;
  p.R = d.R;
  p.S = d.S;
  p.RS = d.R * d.S;
  if (p.RS > kMaxTaps) return CONV2D_ERR_UNSUPPORTED;
  const int CHUNK = d.dt == 0 ? 4 : 8;
  const int ESZ = d.dt == 0 ? 4 : 2;
  const int BUFP = d.dt == 0 ? 32 : 64;  // positions per 32-column TMEM buffer
  const int mh = (d.dh * (d.R - 1)) / d.sh, mw = (d.dw * (d.S - 1)) / d.sw;
  p.NK = d.K <= 16 ? 16 : std::min(round_up(d.K, 32), 256);
  p.n_ntiles = (d.K + p.NK - 1) / p.NK;
  // Copy-engine staging: unit column stride, rows and planes of whole 16-byte chunks, aligned
  // tensors.  Its linear row width WL covers the output columns plus the filter overhang and
  // every pixel of an image row shifted by delta (the row copy starts at -align(pad_w)); at
  // most 256 (one copy box).  Row-tap sharing (unit stride, 32 or more channels, two or more
  // filter rows, room in TMEM for two row taps) takes WL a multiple of 2 CHUNK (an MMA's
  // chunk pair never straddles a dy ring row) and pads the x ring rows to WL + CHUNK; without
  // it WL itself is CHUNK mod 2 CHUNK.  Either way the x ring pitch is CHUNK mod 2 CHUNK, so
  // 16-byte reads of 8 consecutive channel rows fall in distinct banks.
  bool tma = allow_tma && d.sw == 1 && d.W % CHUNK == 0 && d.Q % CHUNK == 0 && ((uintptr_t)x & 15) == 0 &&
             ((uintptr_t)dy & 15) == 0 && encode_tiled_fn() != nullptr;
  p.TRU = 1;
  if (tma && allow_rowshare && d.sh == 1 && d.C >= 32 && d.R > 1 && 2 * p.NK <= 384)
    p.TRU = std::min(std::min(d.R, 4), 384 / p.NK);
  if (allow_rowshare && p.TRU == 1) return CONV2D_ERR_UNSUPPORTED;  // the caller plans without sharing
  if (tma) {
    p.delta = round_up(d.pw, CHUNK) - d.pw;
    int wl = std::max(d.Q + mw, d.W + round_up(d.pw, CHUNK));
    if (p.TRU > 1) {
      wl = round_up(wl, 2 * CHUNK);
      p.WLx = wl + CHUNK;
    } else {
      while (wl % (2 * CHUNK) != CHUNK) ++wl;
      p.WLx = wl;
    }
    p.WL = wl;
    tma = p.WLx <= 256 && 8 * (wl - (d.Q + mw)) <= 2 * wl;  // at most a quarter of the work wasted
  }
  if (!tma && p.TRU > 1) return CONV2D_ERR_UNSUPPORTED;
  if (!tma) {
    // Linear row width: a multiple of the chunk when that wastes at most 1/8 of it, or at
    // most half of it when the output rows are whole chunks, since then it turns the dy
    // staging from one copy per element into 16-byte copies, and the element copies, not
    // the MMAs, pace these plans.
    p.delta = 0;
    const int wl = round_up(d.Q + mw, CHUNK);
    const int waste = wl - (d.Q + mw);
    p.WL = (8 * waste <= wl || (d.Q % CHUNK == 0 && 2 * waste <= wl)) ? wl : d.Q + mw;
    p.WLx = p.WL;
  }
  p.EL = d.P + mh;
  p.Mtot = (long long)d.N * p.EL * p.WL;
  p.tru_step = d.dh;  // (unit row stride only: sh == 1 whenever TRU > 1)
  p.Mit = p.Mtot + (long long)(p.TRU - 1) * p.tru_step * p.WL;
  if (p.Mit >= (1ll << 31)) return CONV2D_ERR_TOO_LARGE;
  p.fd_img = make_fastdiv((uint32_t)(p.EL * p.WL));
  p.fd_WL = make_fastdiv((uint32_t)p.WL);
  p.npl = d.sh * d.sw;
  p.pl_step_h = d.sh;
  p.pl_step_w = d.sw;
  for (int a = 0; a < d.sh; ++a)
    for (int c = 0; c < d.sw; ++c) {
      p.pl_off_h[a * d.sw + c] = a - d.ph;
      p.pl_off_w[a * d.sw + c] = c - d.pw;
    }
  for (int r = 0; r < d.R; ++r)
    for (int s = 0; s < d.S; ++s) {
      const int t = r * d.S + s;
      const int re = r * d.dh, se = s * d.dw;  // the tap's place in the dilated window
      p.tap_plane[t] = (re % d.sh) * d.sw + (se % d.sw);
      p.tap_off[t] = (re / d.sh) * p.WL + se / d.sw;
      p.tap_rc[t] = ((re / d.sh) << 16) | (se / d.sw);
    }
  p.vec_dy = d.Q % CHUNK == 0 && p.WL % CHUNK == 0 && ((uintptr_t)dy & 15) == 0;
  // Row units of 32 TMEM lanes: 32 channels of one tap, or (C < 32) TPU taps x C channels.
  p.Cg = d.C >= 32 ? 32 : d.C;
  p.TPU = d.C >= 32 ? 1 : 32 / d.C;
  p.max_off = 0;
  if (p.TPU == 1) {
    // units of a channel group: (row block rb, column s), base tap (rb * TRU, s)
    const int nrb = (d.R + p.TRU - 1) / p.TRU;
    p.upc = nrb * d.S;
    for (int rb = 0; rb < nrb; ++rb)
      for (int s = 0; s < d.S; ++s) {
        const int t = (rb * p.TRU) * d.S + s;
        p.unit_tap[rb * d.S + s] = t;
        p.max_off = std::max(p.max_off, p.tap_off[t]);
      }
  } else {
    p.upc = (p.RS + p.TPU - 1) / p.TPU;
    for (int t = 0; t < p.RS; ++t) p.max_off = std::max(p.max_off, p.tap_off[t]);
  }
  p.fd_upc = make_fastdiv((uint32_t)p.upc);
  const int ncg = (d.C + p.Cg - 1) / p.Cg;
  p.nunits = ncg * p.upc;
  p.n_mtiles = (p.nunits + 3) / 4;
  // m-tiles per CTA tile: as many accumulators (TRU per m-tile) as TMEM holds next to the 4
  // A buffers, so x and dy are staged once for all of them; two accumulator sets when they fit.
  const int accw = p.TRU * p.NK;
  p.G = std::max(1, std::min(std::min(p.n_mtiles, (512 - 128) / accw), 8));
  p.n_mgroups = (p.n_mtiles + p.G - 1) / p.G;
  p.G = (p.n_mtiles + p.n_mgroups - 1) / p.n_mgroups;  // balance the groups
  p.accb = (128 + 2 * p.G * accw <= 512) ? 2 : 1;
  p.tmem_cols = 32;
  while (p.tmem_cols < 128 + p.accb * p.G * accw) p.tmem_cols <<= 1;
  p.xch = 0;
  for (int mg = 0; mg < p.n_mgroups; ++mg) {
    const int u0 = 4 * p.G * mg, u1 = std::min(p.nunits, 4 * p.G * (mg + 1)) - 1;
    const int cg0 = u0 / p.upc, cg1 = u1 / p.upc;
    p.xch = std::max(p.xch, std::min(d.C, (cg1 + 1) * p.Cg) - cg0 * p.Cg);
  }
  // 16-byte x loads: unit column stride, rows and planes of whole chunks, aligned base;
  // sigma puts the start of every slot group on a chunk-aligned pixel.
  p.vec_x = d.sw == 1 && p.WL % CHUNK == 0 && d.W % CHUNK == 0 && ((uintptr_t)x & 15) == 0;
  p.sigma = p.vec_x ? (CHUNK - d.pw % CHUNK) % CHUNK : 0;
  // x by whole-row tensor copies (1), else by bulk copies of pixel runs when 16-byte aligned (2)
  p.use_tma = tma ? 1 : (p.vec_x && p.vec_dy ? 2 : 0);
  p.xr = round_up(p.xch, 32);
  // Pipeline: the most positions in flight (stages x KB) that fit, then the larger KB.
  bool fitted = false;
  long long best = -1;
  WgradPlan bestp = p;
  for (int KB : {256, 192, 128, 96, 64, 32}) {
    if (KB % BUFP) continue;
    for (int S = 4; S >= 2; --S) {
      WgradPlan q = p;
      q.KB = KB;
      q.stages = S;
      // the ring holds S stages plus the halo, plus a slot group rewritten at each end;
      // row stride: 16 bytes past a multiple of 128 (conflict-free 16-byte reads of 8 rows)
      q.rlen = round_up(S * KB + p.max_off + 2 * CHUNK, 32);
      q.xs = q.rlen;
      while ((q.xs * ESZ) % 128 != 16) q.xs += CHUNK;
      // row ring: S stages plus the halo, plus a row at each end
      q.NR = (S * KB + p.max_off + p.delta + p.WL - 1) / p.WL + 2;
      // dy row ring (row-tap sharing): the rows of S stages plus (TRU - 1) * tru_step rows before
      q.NRd = p.TRU > 1 ? (S * KB + (p.TRU - 1) * p.tru_step * p.WL - 1) / p.WL + 2 : 0;
      q.a_stage_bytes = p.TRU > 1 ? 0 : KB * p.NK * ESZ;
      if (wgrad_smem_bytes(q, d.dt) > di.smem_optin) continue;
      const long long score = (long long)S * KB * 4 + KB / 32;
      if (score > best) {
        best = score;
        bestp = q;
        fitted = true;
      }
    }
  }
  if (!fitted) return CONV2D_ERR_UNSUPPORTED;
  p = bestp;
  p.fd_EL = make_fastdiv((uint32_t)p.EL);
  p.fd_rlen = make_fastdiv((uint32_t)p.rlen);
  p.fd_NR = make_fastdiv((uint32_t)p.NR);
  p.fd_NRd = make_fastdiv((uint32_t)std::max(p.NRd, 1));
  // (sizing calls pass no tensors: their plan assumes the maps encode)
  const bool sizing = x == nullptr && dy == nullptr;
  if (p.use_tma == 1 && !sizing &&
      !((p.TRU > 1 ? encode_dy_row_map(&p.tm_dyr, dy, d.dt, d.N, d.K, d.P, d.Q, p.NK, p.WL, p.dy_nstride)
                   : encode_dy_map(&p.tm_dy, dy, d.dt, d.N, d.K, d.P, d.Q, p.NK, p.dy_nstride)) &&
        encode_x_map(&p.tm_x, x, d.dt, d.N, d.C, d.H, d.W, p.WLx, p.x_nstride))) {
    // The row ring cannot be encoded: plan without sharing, or the slot ring (another linear
    // row width).
    return CONV2D_ERR_UNSUPPORTED;
  }
  if (p.use_tma == 2 && !sizing && !encode_dy_map(&p.tm_dy, dy, d.dt, d.N, d.K, d.P, d.Q, p.NK, p.dy_nstride))
    p.use_tma = 0;  // same ring, staged with cp.async
  // Split the positions so that the tiles fill the SMs with the shortest makespan
  // (tiles per CTA x positions per tile), preferring fewer splits.
  const long long base = (long long)p.n_mgroups * p.n_ntiles;
  const long long stage_count = (p.Mit + p.KB - 1) / p.KB;
  const size_t per_split = (size_t)p.RS * d.C * d.K * sizeof(float);
  long long nsb = 1;
  double best_t = -1.0;
  for (long long ns = 1; ns <= std::min<long long>(stage_count, 4 * (long long)di.sms); ++ns) {
    if (per_split * (size_t)ns > kWorkspaceCap) break;
    const long long slen = (stage_count + ns - 1) / ns;  // stages per split
    const long long waves = (base * ns + di.sms - 1) / di.sms;
    const double tmake = (double)waves * (double)(slen * p.KB + p.max_off + 4 * p.KB);
    if (best_t < 0 || tmake < best_t * 0.98) {
      best_t = tmake;
      nsb = ns;
    }
  }
  long long slen = (stage_count + nsb - 1) / nsb * p.KB;
  p.split_len = slen;
  p.nsplit = (int)((p.Mit + slen - 1) / slen);
  p.total_tiles = base * p.nsplit;
  b.partial_bytes = per_split * (size_t)p.nsplit;
  if (b.partial_bytes > kWorkspaceCap) return CONV2D_ERR_UNSUPPORTED;
  ReducePlan& rp = b.rp;
  rp.partial = p.partial;
  rp.dw = dw;
  rp.K = d.K;
  rp.C = d.C;
  rp.R = d.R;
  rp.S = d.S;
  rp.nsplit = p.nsplit;
  rp.k_pad = d.K;
  rp.c_pad = d.C;
  rp.beta = 0.f;
  rp.flip = 0;
  rp.R_out = d.R;
  rp.S_out = d.S;
  rp.r0 = rp.s0 = 0;
  rp.rstep = rp.sstep = 1;
  rp.gk = rp.gc = 0;
  b.grid = (int)std::min<long long>(p.total_tiles, di.sms);
  return CONV2D_OK;
}

// Backward-filter plan: copy-engine staging when the shape allows it and its row ring fits,
// else the cp.async staging.
// Staging variants of the backward-filter plan, most preferred first: copy-engine row ring
// with row-tap sharing, copy-engine row ring, slot ring.
constexpr bool kWgradVariants[3][2] = {{true, true}, {true, false}, {false, false}};

int build_bwd_filter(const Desc& d, const void* x, const void* dy, void* dw, void* ws, const DevInfo& di,
                     WgradBuild& b) {
  int rc = CONV2D_ERR_UNSUPPORTED;
  for (const auto& v : kWgradVariants) {
    rc = build_bwd_filter_impl(d, x, dy, dw, ws, di, b, v[0], v[1]);
    if (rc != CONV2D_ERR_UNSUPPORTED) return rc;
  }
  return rc;
}

// ---------------------------------------------------------------- strided backward-filter
// With stride st > 1 the filter rows split by the residue rho of the input row they read:
// row p*st - pad + r = st*(p + alpha) + rho.  Phase rho holds the taps r = r0 + st*r'
// (r' < n) with (r - pad - rho) divisible by st; on the plane of input rows congruent to rho
// they read plane row p - pad' + r', pad' = -(r0 - pad - rho) / st >= 0 (r0 < st).  Columns
// likewise.  Every phase is a stride-1 problem over unit-stride planes, so x is copied once
// into the planes (space to depth) and each phase runs the stride-1 backward-filter, whose
// reduce places tap (r', s') at (r0 + sh*r', s0 + sw*s').  Every tap is in one phase, so the
// phases' FLOP add up to the original.  Dilation 1 only.
struct StridePhase {
  int rho, r0, n, pad;
};

std::vector<StridePhase> stride_phases(int R, int pad, int st) {
  std::vector<StridePhase> v;
  for (int rho = 0; rho < st; ++rho) {
    StridePhase f{rho, -1, 0, 0};
    for (int r = 0; r < R; ++r)
      if (((r - pad - rho) % st + st) % st == 0) {
        if (f.n++ == 0) f.r0 = r;
      }
    if (f.n > 0) {
      f.pad = -floor_div(f.r0 - pad - rho, st);
      v.push_back(f);
    }
  }
  return v;
}

size_t align_ws(size_t b);

struct PhaseLayout {
  bool on = false;
  int Hp = 0, Wp = 0;    // plane extent (Wp a whole number of 16-byte chunks)
  size_t xs_bytes = 0;   // planes of all channels (aligned)
  std::vector<StridePhase> rows, cols;
};

// dg: the per-group descriptor; the planes hold all dg.g * dg.C channels.
PhaseLayout phase_layout(const Desc& dg) {
  PhaseLayout L;
  if ((dg.sh == 1 && dg.sw == 1) || dg.dh != 1 || dg.dw != 1) return L;
  const int CHUNK = dg.dt == 0 ? 4 : 8;
  const size_t esz = dg.dt == 0 ? 4 : 2;
  L.on = true;
  L.Hp = ceil_div_i(dg.H, dg.sh);
  L.Wp = round_up(ceil_div_i(dg.W, dg.sw), CHUNK);
  L.xs_bytes = align_ws((size_t)dg.N * dg.sh * dg.sw * dg.g * dg.C * L.Hp * L.Wp * esz);
  L.rows = stride_phases(dg.R, dg.ph, dg.sh);
  L.cols = stride_phases(dg.S, dg.pw, dg.sw);
  return L;
}

// The stride-1 descriptor of phase (a, b): planes as the input, the phase's taps and pads,
// the caller's output extent (P, Q stay; they need not follow from the plane size).
Desc phase_desc(const Desc& dg, const PhaseLayout& L, const StridePhase& a, const StridePhase& b) {
  Desc q = dg;
  q.H = L.Hp;
  q.W = L.Wp;
  q.R = a.n;
  q.S = b.n;
  q.ph = a.pad;
  q.pw = b.pad;
  q.sh = q.sw = 1;
  q.xg = dg.g * dg.sh * dg.sw;
  return q;
}

// Address of the plane of phase (a, b) for group gi within the planes buffer.
const void* phase_plane(const void* xs, const Desc& dg, const PhaseLayout& L, const StridePhase& a,
                        const StridePhase& b, int gi) {
  const size_t esz = dg.dt == 0 ? 4 : 2;
  const size_t pl = (size_t)a.rho * dg.sw + b.rho;
  return byte_ptr(xs) + ((pl * dg.g + gi) * dg.C) * (size_t)L.Hp * L.Wp * esz;
}

// Staging work of a backward-filter plan, in copies: for every (m-group, n-tile) pass over
// the positions, each position stages the x channels of every plane and the dy rows of the
// n tile; a 16-byte (or whole-row tensor) copy counts once, an element copy once per element.
// The stride phases trade element copies of x for one more pass over dy per phase, which
// pays only where x staging dominates (many channels) -- not on a 3-channel stem.
double staging_copies(const WgradPlan& p, int dt) {
  const int CHUNK = dt == 0 ? 4 : 8;
  const double xc = (double)p.xch * p.npl / ((p.vec_x || p.use_tma == 1) ? CHUNK : 1);
  const double dc = (double)p.NK / ((p.vec_dy || p.use_tma == 1) ? CHUNK : 1);
  return (double)p.n_mgroups * p.n_ntiles * (xc + dc) * (double)p.Mit;
}

// True when the phases stage less than the problem as a whole (or it has no plan).
bool phases_stage_less(const std::vector<WgradBuild>& phases, const WgradPlan* whole, int dt) {
  if (whole == nullptr) return true;
  double cp = 0.0;
  for (const WgradBuild& wb : phases) cp += staging_copies(wb.p, dt);
  return cp < staging_copies(*whole, dt);
}

// Plans every phase of group gi (cached); false if one of them has no plan.
int plan_phases(const Desc& dg, const PhaseLayout& L, const void* xs, const void* dyg, void* dwg, void* partial_ws,
                int gi, const DevInfo& di, std::vector<WgradBuild>& out);

// ------------------------------------------------------------------ bf16 channel-chunked wgrad
// Backward-filter of bf16 tensors on channel-chunked planes (WgradMnPlan): x is packed once per
// stride phase plane and dy once into zero-padded planes of the position space
// L = n*EX*WL + e*WL + f, where every filter tap is an offset; the GEMM then stages both operands
// with tensor copies.  Applies to bf16 tensors with unit stride (any dilation) or dilation 1
// (stride phases).  Workspace: the packed x planes, the packed dy, the split partials.
struct MnBuild {
  WgradMnPlan p;
  NhwcPackPlan px, pd;
  ReduceTPlan rp;
  size_t xq_bytes = 0, dyq_bytes = 0, partial_bytes = 0;
  int grid = 0;
};

// One filter dimension split into phases: the taps of a phase read padded plane row e + off of
// a plane whose row e is source row step*e + xoff.  Unit stride: one phase, offsets r*dil,
// xoff = -pad.  Stride st > 1 (dilation 1): the stride phases, offsets r'.
struct MnPhase {
  int xoff;
  std::vector<int> tap, off;  // filter index and its offset
};

std::vector<MnPhase> mn_phases(int R, int pad, int st, int dil) {
  std::vector<MnPhase> v;
  if (st == 1) {
    MnPhase p;
    p.xoff = -pad;
    for (int r = 0; r < R; ++r) {
      p.tap.push_back(r);
      p.off.push_back(r * dil);
    }
    v.push_back(p);
    return v;
  }
  for (const StridePhase& f : stride_phases(R, pad, st)) {
    MnPhase p;
    p.xoff = f.rho - st * f.pad;
    for (int i = 0; i < f.n; ++i) {
      p.tap.push_back(f.r0 + st * i);
      p.off.push_back(i);
    }
    v.push_back(p);
  }
  return v;
}

// Packed planes as dense tensors of 8-byte elements (rank 1 to 4, dims[0] contiguous), two per
// position: either dims[0] = 2 * positions, then chunks (and planes), the box's first dim a run
// of positions; or dims = (2, positions, chunks, planes), the box a run of whole positions.
bool encode_mn_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint32_t* box) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  if (rank < 1 || rank > 4) return false;
  cuuint64_t gd[4], gs[3];
  cuuint32_t bx[4], es[4] = {1u, 1u, 1u, 1u};
  uint64_t stride = 8;  // bytes per element
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    if (i > 0) gs[i - 1] = stride;
    stride *= dims[i];
  }
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, (cuuint32_t)rank, const_cast<void*>(base), gd, gs, bx, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The tap GEMM's view of packed source planes at `base` (nchunk chunks, npl planes, p.Mtot
// positions each), in the form the plan's producers copy it: with a_one, (2, positions, chunks,
// planes) and a box of every row, chunk and plane of a stage; else (2 * positions, chunks,
// planes) and a box of a_box rows.  Every encode of p.tm_src goes through here, so the map and
// the copies the kernel issues always agree.
bool encode_tap_src_map(TapPlan& p, const void* base, int nchunk, int npl, int dt) {
  if (p.a_one) {
    const uint64_t dims[4] = {2, (uint64_t)p.Mtot, (uint64_t)nchunk, (uint64_t)npl};
    const uint32_t box[4] = {2u, (uint32_t)p.rows, (uint32_t)(p.CB / (dt == 0 ? 4 : 8)),
                             p.plane_per_phase ? 1u : (uint32_t)npl};
    return encode_mn_map(&p.tm_src, base, 4, dims, box);
  }
  const uint64_t dims[3] = {2 * (uint64_t)p.Mtot, (uint64_t)nchunk, (uint64_t)npl};
  const uint32_t box[3] = {2 * (uint32_t)p.a_box, 1u, 1u};
  return encode_mn_map(&p.tm_src, base, 3, dims, box);
}

// Work-unit tiling of a pack (NhwcPackPlan): the most padded rows per unit whose staged channel
// runs of one chunk fit 32 KB of shared memory (at least one row, then up to 200 KB), then the
// chunks per unit; false if none fits or the unit count passes 32 bits.
bool setup_pack_tiles(NhwcPackPlan& q, int esz) {
  const int CHUNK = 16 / esz;
  int lo = q.off_h[0], hi = q.off_h[0];
  for (int pl = 1; pl < q.npl; ++pl) {
    lo = std::min(lo, q.off_h[pl]);
    hi = std::max(hi, q.off_h[pl]);
  }
  q.off_h_min = lo;
  q.h_span = hi - lo;
  auto pitch = [&](int te) {  // elements per staged channel run, rounded up to 16 bytes
    const long long rows = std::min<long long>((long long)(te - 1) * q.step_h + q.h_span + 1, q.H);
    return (rows * q.W * esz + 15) / 16 * 16 / esz;
  };
  int te = 1;
  while (te < q.EX && (long long)CHUNK * pitch(te + 1) * esz <= 32 * 1024) ++te;
  if ((long long)CHUNK * pitch(te) * esz > 200 * 1024) return false;
  q.te = te;
  q.ch_pitch = (int)pitch(te);
  q.n_etiles = (q.EX + te - 1) / te;
  // chunks per unit: as many as fit the same 32 KB, while the units still number four per SM
  // of a full GPU (small images: one unit per chunk leaves the work per block too small)
  int cg = 1;
  while (cg < q.nchunk && (long long)(cg + 1) * CHUNK * q.ch_pitch * esz <= 32 * 1024 &&
         (long long)q.N * ((q.nchunk + cg) / (cg + 1)) * q.n_etiles >= 4 * 152)
    ++cg;
  q.cg = cg;
  q.ngroups = (q.nchunk + cg - 1) / cg;
  const long long units = (long long)q.N * q.ngroups * q.n_etiles;
  if (units >= (1ll << 31)) return false;
  q.units = (unsigned)units;
  q.fd_et = make_fastdiv((uint32_t)q.n_etiles);
  q.fd_ng = make_fastdiv((uint32_t)q.ngroups);
  return true;
}

int build_wgrad_mn(const Desc& d, const void* x, const void* dy, void* dw, void* ws, const DevInfo& di, MnBuild& b) {
  if (d.dt != CONV2D_DTYPE_BF16) return CONV2D_ERR_UNSUPPORTED;
  if (d.R * d.S > kMaxTaps) return CONV2D_ERR_UNSUPPORTED;  // the plan's tap tables
  if ((d.sh > 1 || d.sw > 1) && (d.dh != 1 || d.dw != 1)) return CONV2D_ERR_UNSUPPORTED;
  if (d.K % 4 != 0) return CONV2D_ERR_UNSUPPORTED;  // the reduce reads 4 output channels at a time
  const std::vector<MnPhase> rows = mn_phases(d.R, d.ph, d.sh, d.dh), cols = mn_phases(d.S, d.pw, d.sw, d.dw);
  int mo_r = 0, mo_c = 0;
  for (const MnPhase& a : rows)
    for (int o : a.off) mo_r = std::max(mo_r, o);
  for (const MnPhase& c : cols)
    for (int o : c.off) mo_c = std::max(mo_c, o);
  const int EX = d.P + mo_r, WL = d.Q + mo_c;
  const long long Mtot = (long long)d.N * EX * WL;
  if (Mtot >= (1ll << 31)) return CONV2D_ERR_TOO_LARGE;
  const int npl = (int)(rows.size() * cols.size());
  if (npl > kMaxPlanes) return CONV2D_ERR_UNSUPPORTED;
  WgradMnPlan& p = b.p;
  std::memset(&p, 0, sizeof(p));
  p.C = d.C;
  p.K = d.K;
  p.RS = d.R * d.S;
  p.Mtot = Mtot;
  p.NK = d.K >= 256 ? 256 : std::max(16, round_up(d.K, 16));
  p.n_ktiles = (d.K + p.NK - 1) / p.NK;
  p.n_ctiles = (d.C + 127) / 128;
  // taps of every plane, sorted by offset
  struct Tap {
    int off, out;
  };
  std::vector<std::vector<Tap>> ptaps((size_t)npl);
  int maxtaps = 1;
  for (size_t a = 0; a < rows.size(); ++a)
    for (size_t c = 0; c < cols.size(); ++c) {
      std::vector<Tap>& v = ptaps[a * cols.size() + c];
      for (size_t i = 0; i < rows[a].tap.size(); ++i)
        for (size_t j = 0; j < cols[c].tap.size(); ++j)
          v.push_back({rows[a].off[i] * WL + cols[c].off[j], rows[a].tap[i] * d.S + cols[c].tap[j]});
      std::stable_sort(v.begin(), v.end(), [](const Tap& u, const Tap& w) { return u.off < w.off; });
      maxtaps = std::max(maxtaps, (int)v.size());
    }
  p.T = std::max(1, std::min(maxtaps, 512 / p.NK));
  p.tmem_cols = 32;
  while (p.tmem_cols < p.T * p.NK) p.tmem_cols <<= 1;
  const size_t budget = di.smem_optin - 2048;
  // Candidate stage lengths; each groups every plane's taps greedily (at most T taps whose
  // offsets fit one copy box with the stage).  Preferred: the fewest groups (every group stages
  // dy and x again), then at least 3 pipeline stages, then the longer stage.
  bool fitted = false;
  WgradMnPlan best = p;
  long long best_score = -1;
  for (int KB : {128, 64, 32}) {
    WgradMnPlan q = p;
    int ng = 0, nt = 0, span = 0;
    bool ok = true;
    for (int pl = 0; pl < npl && ok; ++pl) {
      const std::vector<Tap>& v = ptaps[(size_t)pl];
      for (size_t i = 0; i < v.size();) {
        if (ng >= kMaxTaps) {
          ok = false;
          break;
        }
        size_t j = i + 1;
        while (j < v.size() && (int)(j - i) < q.T && v[j].off - v[i].off + KB <= 128) ++j;
        q.grp_plane[ng] = pl;
        q.grp_tap0[ng] = nt;
        q.grp_ntaps[ng] = (int)(j - i);
        q.grp_off0[ng] = v[i].off;
        for (size_t u = i; u < j; ++u, ++nt) {
          q.tap_delta[nt] = v[u].off - v[i].off;
          q.tap_out[nt] = v[u].out;
        }
        span = std::max(span, v[j - 1].off - v[i].off);
        ++ng;
        i = j;
      }
    }
    if (!ok || KB + span > 128) continue;  // a copy box row is at most 128 positions (256 elements)
    const int KBX = KB + span;
    const int a_box = 16 * KBX * 16, b_box = (q.NK / 8) * KB * 16;
    const int a_st = round_up(a_box, 1024), b_st = round_up(b_box, 1024);
    const size_t fixed = 8 * (2 * 8 + 3) + 16 + 1024 + 8 * 32 * 80;  // barriers, epilogue staging
    long long st = ((long long)budget - (long long)fixed) / (a_st + b_st);
    if (st > 4) st = 4;
    if (st < 2) continue;
    q.ngroups = ng;
    q.KB = KB;
    q.KBX = KBX;
    q.stages = (int)st;
    q.a_stage_bytes = a_st;
    q.b_stage_bytes = b_st;
    q.tx_bytes = a_box + b_box;
    if (wgrad_mn_smem_bytes(q) > di.smem_optin) continue;
    const long long score = (long long)(kMaxTaps + 1 - ng) * 1000000 + (st >= 3 ? 1000 : 0) + KB;
    if (score > best_score) {
      best_score = score;
      best = q;
      fitted = true;
    }
  }
  if (fitted) p = best;
  if (!fitted) return CONV2D_ERR_UNSUPPORTED;
  // splits: one wave of tiles when there are fewer tile shapes than SMs
  const long long base = (long long)p.ngroups * p.n_ctiles * p.n_ktiles;
  const long long stage_count = (Mtot + p.KB - 1) / p.KB;
  long long ns = base >= di.sms ? 1 : std::max(1ll, (long long)di.sms / base);
  ns = std::min(ns, stage_count);
  const size_t per_split = (size_t)p.RS * d.C * d.K * sizeof(float);
  while (ns > 1 && per_split * (size_t)ns > kWorkspaceCap / 2) --ns;
  p.split_len = (stage_count + ns - 1) / ns * p.KB;
  p.nsplit = (int)((Mtot + p.split_len - 1) / p.split_len);
  p.total_tiles = base * p.nsplit;
  b.grid = (int)std::min<long long>(p.total_tiles, di.sms);
  // workspace: packed x planes, packed dy, partials
  const int C8 = (d.C + 7) / 8, K8 = (d.K + 7) / 8;
  b.xq_bytes = (size_t)npl * C8 * (size_t)Mtot * 16;
  b.dyq_bytes = (size_t)K8 * (size_t)Mtot * 16;
  b.partial_bytes = per_split * (size_t)p.nsplit;
  if (align_ws(b.xq_bytes) + align_ws(b.dyq_bytes) + b.partial_bytes > kWorkspaceCap) return CONV2D_ERR_UNSUPPORTED;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  void* xq = w8 ? w8 : nullptr;
  void* dyq = w8 ? w8 + align_ws(b.xq_bytes) : nullptr;
  p.partial = w8 ? reinterpret_cast<float*>(w8 + align_ws(b.xq_bytes) + align_ws(b.dyq_bytes)) : nullptr;
  // packs
  NhwcPackPlan& px = b.px;
  std::memset(&px, 0, sizeof(px));
  px.src = x;
  px.dst = xq;
  px.src_nstride = (long long)d.g * d.C * d.H * d.W;
  px.N = d.N;
  px.C = d.C;
  px.H = d.H;
  px.W = d.W;
  px.nchunk = C8;
  px.EX = EX;
  px.WL = WL;
  px.fd_WL = make_fastdiv((uint32_t)WL);
  px.npl = npl;
  px.step_h = d.sh;
  px.step_w = d.sw;
  for (size_t a = 0; a < rows.size(); ++a)
    for (size_t c = 0; c < cols.size(); ++c) {
      px.off_h[a * cols.size() + c] = rows[a].xoff;
      px.off_w[a * cols.size() + c] = cols[c].xoff;
    }
  NhwcPackPlan& pd = b.pd;
  std::memset(&pd, 0, sizeof(pd));
  pd.src = dy;
  pd.dst = dyq;
  pd.src_nstride = (long long)d.g * d.K * d.P * d.Q;
  pd.N = d.N;
  pd.C = d.K;
  pd.H = d.P;
  pd.W = d.Q;
  pd.nchunk = K8;
  pd.EX = EX;
  pd.WL = WL;
  pd.fd_WL = make_fastdiv((uint32_t)WL);
  pd.npl = 1;
  pd.step_h = pd.step_w = 1;
  if ((long long)EX * WL >= (1ll << 31)) return CONV2D_ERR_TOO_LARGE;
  if (!setup_pack_tiles(px, 2) || !setup_pack_tiles(pd, 2)) return CONV2D_ERR_UNSUPPORTED;
  // tensor maps over the packed planes (sizing calls pass no workspace)
  if (w8 != nullptr) {
    const uint64_t xd[3] = {2 * (uint64_t)Mtot, (uint64_t)C8, (uint64_t)npl};
    const uint32_t xb[3] = {2 * (uint32_t)p.KBX, 16, 1};
    const uint64_t yd[2] = {2 * (uint64_t)Mtot, (uint64_t)K8};
    const uint32_t yb[2] = {2 * (uint32_t)p.KB, (uint32_t)(p.NK / 8)};
    if (!encode_mn_map(&p.tm_x, xq, 3, xd, xb) || !encode_mn_map(&p.tm_dy, dyq, 2, yd, yb))
      return CONV2D_ERR_UNSUPPORTED;
  }
  ReduceTPlan& rp = b.rp;
  std::memset(&rp, 0, sizeof(rp));
  rp.partial = p.partial;
  rp.dw = dw;
  rp.rows = d.C * d.R * d.S;
  rp.K = d.K;
  rp.RS = d.R * d.S;
  rp.nsplit = p.nsplit;
  return CONV2D_OK;
}

size_t mn_ws_bytes(const MnBuild& b) {
  return align_ws(b.xq_bytes) + align_ws(b.dyq_bytes) + align_ws(b.partial_bytes);
}

int check_ptrs(const void* a, const void* b, const void* c, int dt) {
  if (!a || !b || !c) return CONV2D_ERR_NULLPTR;
  const uintptr_t m = dt == CONV2D_DTYPE_F32 ? 3 : 1;
  if (((uintptr_t)a & m) || ((uintptr_t)b & m) || ((uintptr_t)c & m)) return CONV2D_ERR_ALIGN;
  return CONV2D_OK;
}

// Workspace of the bias-gradient sums of conv2d_bwd_filter_ex: fp32 partials per (channel,
// image) for the K sums over dy and the C sums over x, each region 256-byte aligned.
size_t align_ws(size_t b) { return (b + 255) & ~size_t(255); }

// Images per block of a channel sum: enough that a block reads about 64 KB (at least one
// image), fewer while the blocks would number under four per SM.  The partials (Ch * nblk
// floats) fit the Ch * N floats the workspace holds for them; a block's 16-byte groups stay
// within 32-bit counts.
void chan_sum_blocks(ChanSumPlan& cp, int dt) {
  const long long img = cp.HW * (dt == 0 ? 4 : 2);
  int ipb = (int)std::max<long long>(1, std::min<long long>(cp.N, (64 * 1024) / std::max<long long>(img, 1)));
  while (ipb > 1 && (long long)ipb * img / 16 >= (1ll << 31)) --ipb;
  while (ipb > 1 && (long long)cp.Ch * ((cp.N + ipb - 1) / ipb) < 4 * 152) ipb = (ipb + 1) / 2;
  cp.ipb = ipb;
  cp.nblk = (cp.N + ipb - 1) / ipb;
}

size_t chan_sum_bytes(const Desc& d) {  // the sums cover all d.g groups' channels
  return align_ws((size_t)d.g * d.K * d.N * sizeof(float)) + align_ws((size_t)d.g * d.C * d.N * sizeof(float));
}

int check_ws(void* ws, size_t have, size_t need) {
  if (need == 0) return CONV2D_OK;
  if (!ws) return CONV2D_ERR_NULLPTR;
  if ((uintptr_t)ws & 15) return CONV2D_ERR_ALIGN;
  if (have < need) return CONV2D_ERR_WORKSPACE;
  return CONV2D_OK;
}

// Kernels this library has enqueued since the process started (conv2d_kernel_launches).
std::atomic<unsigned long long> g_launches{0};

// Status of a launch helper that enqueued `kernels` kernels when it returned cudaSuccess.
int launch_err(cudaError_t e, int kernels = 1) {
  if (e == cudaSuccess) {
    g_launches.fetch_add((unsigned long long)kernels, std::memory_order_relaxed);
    return CONV2D_OK;
  }
  cudaGetLastError();
  return CONV2D_ERR_LAUNCH;
}

// Plans of recent calls.  A plan depends only on the descriptor, the device and the tensor and
// workspace addresses (the tensor maps and the launch parameters embed them), so a call that
// repeats all of these reuses the plan instead of searching tile shapes and encoding tensor
// maps again.  Small, fixed size, replaced round-robin; guarded by a mutex.
struct PlanKey {
  int op, dev;
  Desc d;
  const void* ptr[4];
};

bool same_key(const PlanKey& a, const PlanKey& b) {
  return a.op == b.op && a.dev == b.dev && std::memcmp(&a.d, &b.d, sizeof(Desc)) == 0 && a.ptr[0] == b.ptr[0] &&
         a.ptr[1] == b.ptr[1] && a.ptr[2] == b.ptr[2] && a.ptr[3] == b.ptr[3];
}

// Forward / backward-data as one or more tap-GEMM passes.  The tap GEMM stages, per k-block,
// the filter slices of every tap of a phase; when that does not fit twice in shared memory
// (large filters over many source channels) the taps u = r*S + s are split into contiguous
// ranges, one pass each: the first pass applies the caller's bias and beta, the later ones
// add onto the output (beta = 1).  Each pass has its own repacked filter in the workspace.

// Backward-data for few input channels (dgrad_c2i_kernel): fp32, C <= 8, S <= 8, strides <= 8,
// C*sh <= 16 (the accumulator N, double-buffered in TMEM), the column halo dlt_w <= 7 of 32 dy
// columns, the row halo dlt_h <= 5, the resident filter operand <= 64 KB, everything within
// shared memory.  d is the per-group descriptor.
int build_c2i(const Desc& d, const void* dy, const void* w, void* dx, const DevInfo& di, C2iPlan& p) {
  if (d.dt != CONV2D_DTYPE_F32 || d.C > 8 || d.S > 8 || d.sh > 8 || d.sw > 8 || d.C * d.sh > 16)
    return CONV2D_ERR_UNSUPPORTED;
  const int dlt_h = (d.R - 1) * d.dh / d.sh, dlt_w = (d.S - 1) * d.dw / d.sw;
  if (dlt_h > 5 || dlt_w > 7) return CONV2D_ERR_UNSUPPORTED;
  std::memset(&p, 0, sizeof(p));
  p.dy = dy;
  p.w = w;
  p.dx = dx;
  p.N = d.N;
  p.C = d.C;
  p.H = d.H;
  p.W = d.W;
  p.K = d.K;
  p.R = d.R;
  p.S = d.S;
  p.P = d.P;
  p.Q = d.Q;
  p.sh = d.sh;
  p.sw = d.sw;
  p.ph = d.ph;
  p.pw = d.pw;
  p.dh = d.dh;
  p.dw = d.dw;
  p.dy_nstride = (long long)d.g * d.K * d.P * d.Q;
  p.dx_nstride = (long long)d.g * d.C * d.H * d.W;
  p.Nr = round_up(d.C * d.sh * 8, 16);
  p.nkb = (d.K + 15) / 16;
  p.dlt_h = dlt_h;
  p.dlt_w = dlt_w;
  p.EH = 8 + dlt_h;
  p.TWq = 32 - dlt_w;
  p.p_start = d.ph / d.sh;
  p.q_start = d.pw / d.sw;
  p.ntp = ceil_div_i(d.H + d.ph - p.p_start * d.sh, 8 * d.sh);
  p.ntq = ceil_div_i(d.W + d.pw - p.q_start * d.sw, p.TWq * d.sw);
  p.tiles = (long long)d.N * p.ntp * p.ntq;
  if ((long long)p.ntp * p.ntq >= (1ll << 31)) return CONV2D_ERR_UNSUPPORTED;  // per-image tile index in 32 bits
  const long long bb = (long long)(dlt_h + 1) * p.nkb * 4 * p.Nr * 16;
  if (bb > 64 * 1024) return CONV2D_ERR_UNSUPPORTED;
  p.b_bytes = (int)bb;
  p.a_bytes = 4 * p.EH * 32 * 16;
  int tc = 32;
  while (tc < 4 * p.Nr) tc <<= 1;
  p.tmem_cols = tc;
  // staged operand slots: three if they fit, else two; dy boxes by tensor copies where dy's
  // row and channel strides are 16-byte multiples: three box slots if they fit, else two
  p.nraw = 0;
  p.nast = 3;
  if (c2i_smem_bytes(p) > di.smem_optin) p.nast = 2;
  if (c2i_smem_bytes(p) > di.smem_optin) return CONV2D_ERR_UNSUPPORTED;
  p.nraw_tma = 0;
  if (d.Q % 4 == 0 && ((long long)d.P * d.Q) % 4 == 0)
    for (int nr = 3; nr >= 2; --nr) {
      p.nraw = nr;
      if (c2i_smem_bytes(p) <= di.smem_optin) {
        p.nraw_tma = nr;
        break;
      }
    }
  p.nraw = 0;
  return CONV2D_OK;
}

// dy of one group (Q, P, K, N), fp32, box (36, EH, 16, 1) for dgrad_c2i_kernel.
bool encode_c2i_dy_map(CUtensorMap* m, const void* dy, const C2iPlan& p) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn || ((uintptr_t)dy & 15) != 0) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)p.Q, (cuuint64_t)p.P, (cuuint64_t)p.K, (cuuint64_t)p.N};
  const cuuint64_t strides[3] = {(cuuint64_t)p.Q * 4, (cuuint64_t)p.P * p.Q * 4, (cuuint64_t)p.dy_nstride * 4};
  const cuuint32_t box[4] = {36u, (cuuint32_t)p.EH, 16u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(dy), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct TapSet {
  std::vector<TapBuild> pass;
  size_t pack_bytes = 0;  // workspace for all passes' repacked filters (and the packed source)
};

// packed_src: a single-pass plan may stage its source rows from a channel-chunk packed copy
// of the source, placed in the workspace after the repacked filter (the allocation-free entry
// point passes false: its scratch holds the filter only).
int build_tap_set(int op, const Desc& d, const void* src, const void* w, void* dst, void* ws, const DevInfo& di,
                  TapSet& out, bool packed_src) {
  const int RS = d.R * d.S;
  for (int n = 1; n <= std::min(RS, kMaxTapPasses); ++n) {
    TapSet set;
    size_t off = 0;
    int rc = CONV2D_OK;
    for (int i = 0; i < n; ++i) {
      const int lo = (int)((long long)RS * i / n), hi = (int)((long long)RS * (i + 1) / n);
      void* wsi = ws != nullptr ? static_cast<void*>(static_cast<uint8_t*>(ws) + off) : nullptr;
      TapBuild b;
      const bool pk = packed_src && n == 1;
      rc = op == CONV2D_OP_FWD ? build_fwd(d, src, w, dst, wsi, di, b, n == 1 ? 0 : lo, n == 1 ? 1 << 30 : hi, pk)
                               : build_bwd_data(d, src, w, dst, wsi, di, b, n == 1 ? 0 : lo, n == 1 ? 1 << 30 : hi, pk);
      if (rc != CONV2D_OK) break;
      off += i + 1 < n ? align_ws(b.pack_bytes) : b.pack_bytes;
      set.pass.push_back(b);
    }
    if (rc == CONV2D_OK && n == 1 && set.pass[0].p.a_tma) {
      TapBuild& b = set.pass[0];
      const size_t xoff = align_ws(off);
      off = xoff + b.src_pack_bytes;
      b.px.dst = ws != nullptr ? static_cast<void*>(static_cast<uint8_t*>(ws) + xoff) : nullptr;
      if (ws != nullptr) {  // sizing calls pass no workspace
        if (!encode_tap_src_map(b.p, b.px.dst, b.px.nchunk, b.px.npl, d.dt)) return CONV2D_ERR_UNSUPPORTED;
      }
    }
    if (rc == CONV2D_OK) {
      set.pack_bytes = off;
      out = std::move(set);
      return CONV2D_OK;
    }
    if (rc != CONV2D_ERR_UNSUPPORTED) return rc;
  }
  return CONV2D_ERR_UNSUPPORTED;
}

template <class Build>
struct PlanCache {
  static constexpr int kEntries = 16;
  std::mutex mu;
  PlanKey key[kEntries];
  Build val[kEntries];
  int used = 0, next = 0;
  bool get(const PlanKey& k, Build& out) {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i)
      if (same_key(key[i], k)) {
        out = val[i];
        return true;
      }
    return false;
  }
  void put(const PlanKey& k, const Build& b) {
    std::lock_guard<std::mutex> lk(mu);
    key[next] = k;
    val[next] = b;
    next = (next + 1) % kEntries;
    if (used < kEntries) ++used;
  }
};

PlanCache<TapSet> g_tap_plans;
PlanCache<C2iPlan> g_c2i_plans;
PlanCache<WgradBuild> g_wgrad_plans;
PlanCache<MnBuild> g_mn_plans;
PlanCache<size_t> g_ws_sizes;
constexpr int kMnKey = 17;  // cache key tag of the channel-chunked backward-filter plans (not an op code)
constexpr int kFusedKey = 18;  // cache key tag of the both-gradients plans

int workspace_size_uncached(int op, const Desc& d, size_t* bytes);

PlanKey make_key(int op, const Desc& d, const void* a, const void* b, const void* c, const void* ws) {
  PlanKey k;
  std::memset(static_cast<void*>(&k), 0, sizeof(k));  // padding too: keys compare by memcmp
  k.op = op;
  cudaGetDevice(&k.dev);
  k.d = d;
  k.ptr[0] = a;
  k.ptr[1] = b;
  k.ptr[2] = c;
  k.ptr[3] = ws;
  return k;
}

int plan_phases(const Desc& dg, const PhaseLayout& L, const void* xs, const void* dyg, void* dwg, void* partial_ws,
                int gi, const DevInfo& di, std::vector<WgradBuild>& out) {
  out.clear();
  for (const StridePhase& a : L.rows)
    for (const StridePhase& b : L.cols) {
      const Desc q = phase_desc(dg, L, a, b);
      const void* xq = xs != nullptr ? phase_plane(xs, dg, L, a, b, gi) : nullptr;
      WgradBuild wb;
      const PlanKey key = make_key(CONV2D_OP_BWD_FILTER, q, xq, dyg, dwg, partial_ws);
      if (xs == nullptr || !g_wgrad_plans.get(key, wb)) {
        const int rc = build_bwd_filter(q, xq, dyg, dwg, partial_ws, di, wb);
        if (rc) return rc;
        if (xs != nullptr) g_wgrad_plans.put(key, wb);
      }
      // the phase's taps in the caller's filter
      wb.rp.R_out = dg.R;
      wb.rp.S_out = dg.S;
      wb.rp.r0 = a.r0;
      wb.rp.s0 = b.r0;
      wb.rp.rstep = dg.sh;
      wb.rp.sstep = dg.sw;
      out.push_back(wb);
    }
  return CONV2D_OK;
}

// Workspace of the phase path: the planes, then the largest phase's partials (the phases
// reuse them in stream order), for whichever staging variant a phase ends up with.
int phase_workspace(const Desc& dg, const PhaseLayout& L, const DevInfo& di, size_t& partial) {
  partial = 0;
  for (const StridePhase& a : L.rows)
    for (const StridePhase& b : L.cols) {
      const Desc q = phase_desc(dg, L, a, b);
      WgradBuild wb;
      const int rc = build_bwd_filter(q, nullptr, nullptr, nullptr, nullptr, di, wb);
      if (rc) return rc;
      partial = std::max(partial, wb.partial_bytes);
      for (const auto& v : kWgradVariants) {
        WgradBuild b2;
        if (build_bwd_filter_impl(q, nullptr, nullptr, nullptr, nullptr, di, b2, v[0], v[1]) == CONV2D_OK)
          partial = std::max(partial, b2.partial_bytes);
      }
    }
  return CONV2D_OK;
}

// Workspace the stride phases of dg need (planes, largest partials, bias sums), or 0 when
// they do not apply, do not plan, or would pass the workspace cap (the problem then runs as a
// whole).  The size query and the call both decide from this value.  Cached per descriptor.
constexpr int kPhaseNeedKey = 16;  // cache key tag (not an op code)

size_t phase_need(const Desc& dg, const DevInfo& di) {
  const PhaseLayout L = phase_layout(dg);
  if (!L.on) return 0;
  const PlanKey key = make_key(kPhaseNeedKey, dg, nullptr, nullptr, nullptr, nullptr);
  size_t v = 0;
  if (g_ws_sizes.get(key, v)) return v;
  size_t partial = 0;
  if (phase_workspace(dg, L, di, partial) == CONV2D_OK) {
    v = L.xs_bytes + align_ws(partial) + chan_sum_bytes(dg);
    if (v > kWorkspaceCap) v = 0;
  }
  g_ws_sizes.put(key, v);
  return v;
}

}  // namespace

namespace cg3 {
// Status of a launch made by another file of the library (the 3-D layout copies), counted
// like this file's launches.
int count_launch(cudaError_t e, int kernels) { return launch_err(e, kernels); }
}  // namespace cg3

extern "C" {

int conv2d_output_dim(int in, int pad, int k, int stride, int* out) {
  if (!out || in <= 0 || k <= 0 || pad < 0 || stride < 1) return CONV2D_ERR_BAD_DESC;
  const int v = out_dim(in, pad, k, stride);
  if (v < 1) return CONV2D_ERR_SHAPE;
  *out = v;
  return CONV2D_OK;
}

int conv2d_workspace_size(int op, int N, int C, int H, int W, int K, int R, int S, int pad_h, int pad_w,
                          int stride_h, int stride_w, int P, int Q, int dtype, size_t* bytes) {
  return conv2d_workspace_size_ex(op, N, C, H, W, K, R, S, pad_h, pad_w, stride_h, stride_w, P, Q, 1, 1, 1, dtype,
                                  bytes);
}

int conv2d_workspace_size_ex(int op, int N, int C, int H, int W, int K, int R, int S, int pad_h, int pad_w,
                             int stride_h, int stride_w, int P, int Q, int dil_h, int dil_w, int groups, int dtype,
                             size_t* bytes) {
  if (!bytes) return CONV2D_ERR_NULLPTR;
  const Desc dt{N, C, H, W, K, R, S, pad_h, pad_w, stride_h, stride_w, P, Q, dtype, dil_h, dil_w};
  int rc = validate(dt);
  if (rc) return rc;
  Desc d;
  rc = group_desc(dt, groups, d);  // per-group plans; the bias sums cover the whole tensors
  if (rc) return rc;
  const PlanKey key = make_key(op, d, nullptr, nullptr, nullptr, nullptr);
  if (g_ws_sizes.get(key, *bytes)) return CONV2D_OK;
  rc = workspace_size_uncached(op, d, bytes);
  if (rc == CONV2D_OK) g_ws_sizes.put(key, *bytes);
  return rc;
}

}  // extern "C"

namespace {
// Both gradients in one call (conv2d_bwd).  bf16, one group: the backward-filter plan packs x
// and dy into channel-chunk planes; when the backward-data plan stages dy from one packed plane
// of the same grid (rows EX, row width WL, dy at its origin), it reads that same pack, so dy is
// read from memory once for both gradients (the pages' backward pass schedules backward-data
// and backward-weights together on the shared output gradient).  Workspace: the
// backward-filter plan's, then the backward-data filter pack.  Otherwise the two ops run one
// after the other in the same workspace.
struct FusedBwd {
  bool fused = false;
  MnBuild mb;
  TapSet set;
  size_t tap_off = 0;  // offset of the backward-data part of the workspace
  size_t need = 0;
};

int build_fused_bwd(const Desc& d, const void* x, const void* w, const void* dy, void* dx, void* dw, void* ws,
                    const DevInfo& di, FusedBwd& f) {
  f.fused = false;
  if (d.dt == CONV2D_DTYPE_BF16 && d.g == 1 && build_wgrad_mn(d, x, dy, dw, ws, di, f.mb) == CONV2D_OK) {
    f.tap_off = align_ws(mn_ws_bytes(f.mb));
    void* wt = ws != nullptr ? static_cast<void*>(static_cast<uint8_t*>(ws) + f.tap_off) : nullptr;
    const int rc = build_tap_set(CONV2D_OP_BWD_DATA, d, dy, w, dx, wt, di, f.set, true);
    if (rc) return rc;
    const TapBuild& b = f.set.pass[0];
    const NhwcPackPlan& q = f.mb.pd;  // dy as the backward-filter plan packs it
    if (f.set.pass.size() == 1 && b.p.a_tma && b.p.npl == 1 && b.p.pl_off_h[0] == 0 && b.p.pl_off_w[0] == 0 &&
        b.p.pl_step_h == 1 && b.p.pl_step_w == 1 && b.p.EL == q.EX && b.p.WL == q.WL && b.px.nchunk == q.nchunk &&
        b.p.Mtot == (long long)q.N * q.EX * q.WL) {
      f.fused = true;
      f.need = f.tap_off + b.pack_bytes;
      if (ws != nullptr) {  // the backward-data copies read the backward-filter plan's dy pack
        if (!encode_tap_src_map(f.set.pass[0].p, q.dst, q.nchunk, 1, d.dt)) return CONV2D_ERR_UNSUPPORTED;
      }
      return CONV2D_OK;
    }
  }
  return CONV2D_OK;
}

PlanCache<FusedBwd> g_fused_plans;

int workspace_size_uncached(int op, const Desc& d, size_t* bytes) {
  int rc;
  const DevInfo di = device_info();
  if (is_depthwise(d) && op != CONV2D_OP_BWD) {  // d: the per-group descriptor (d.g groups)
    Desc t = d;
    t.C = d.C * d.g;
    t.K = d.K * d.g;
    *bytes = op == CONV2D_OP_BWD_FILTER ? align_ws(dw_partial_bytes(dw_plan(t, d, di.sms))) + chan_sum_bytes(d) : 0;
    return CONV2D_OK;
  }
  if (op == CONV2D_OP_BWD) {
    FusedBwd f;
    rc = build_fused_bwd(d, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, di, f);
    if (rc) return rc;
    size_t a = 0, b = 0;
    rc = workspace_size_uncached(CONV2D_OP_BWD_DATA, d, &a);
    if (rc) return rc;
    rc = workspace_size_uncached(CONV2D_OP_BWD_FILTER, d, &b);
    if (rc) return rc;
    *bytes = std::max({a, b, f.fused ? f.need : size_t(0)});
    return CONV2D_OK;
  }
  if (op == CONV2D_OP_FWD || op == CONV2D_OP_BWD_DATA) {  // the choices of run_tap, in its order
    Desc t = d;
    t.C = d.g * d.C;
    t.K = d.g * d.K;
    t.g = 1;
    if (blockdiag_groups(op, t, d.g)) {  // the block-diagonal single pass over the whole tensors
      TapSet whole, per;
      if (build_tap_set(op, t, nullptr, nullptr, nullptr, nullptr, di, whole, true) == CONV2D_OK) {
        // (and room for the per-group passes, should the call's pointers not plan whole)
        const bool per_ok = build_tap_set(op, d, nullptr, nullptr, nullptr, nullptr, di, per, true) == CONV2D_OK;
        *bytes = std::max(whole.pack_bytes, per_ok ? per.pack_bytes : size_t(0));
        return CONV2D_OK;
      }
    }
    C2iPlan cp;
    if (op == CONV2D_OP_BWD_DATA && build_c2i(d, nullptr, nullptr, nullptr, di, cp) == CONV2D_OK) {
      *bytes = 0;
      return CONV2D_OK;
    }
    TapSet set;
    rc = build_tap_set(op, d, nullptr, nullptr, nullptr, nullptr, di, set, true);
    if (rc) return rc;
    *bytes = set.pack_bytes;
    return CONV2D_OK;
  }
  if (op == CONV2D_OP_BWD_FILTER) {
    // bf16: the channel-chunked path when it plans (size for it and for the others)
    size_t mn = 0;
    if (d.dt == CONV2D_DTYPE_BF16) {
      MnBuild mb;
      if (build_wgrad_mn(d, nullptr, nullptr, nullptr, nullptr, di, mb) == CONV2D_OK)
        mn = mn_ws_bytes(mb) + chan_sum_bytes(d);
      if (d.g > 1) {  // grouped: the one pass over the whole tensors (conv2d_bwd_filter_ex)
        Desc t = d;
        t.C = d.g * d.C;
        t.K = d.g * d.K;
        t.g = 1;
        MnBuild mw;
        if (build_wgrad_mn(t, nullptr, nullptr, nullptr, nullptr, di, mw) == CONV2D_OK)
          mn = std::max(mn, mn_ws_bytes(mw) + chan_sum_bytes(d));
      }
    }
    // Strided filters run as stride phases when every phase plans (else as one problem);
    // size for either.
    const size_t phased = std::max(phase_need(d, di), mn);
    // The launch plans the copy-engine staging unless its tensor maps fail to encode for the
    // actual tensors; size for whichever of the two plans it ends up with.
    WgradBuild b;
    rc = build_bwd_filter(d, nullptr, nullptr, nullptr, nullptr, di, b);
    if (rc) return phased ? (*bytes = phased, CONV2D_OK) : rc;
    size_t need = b.partial_bytes;
    for (const auto& v : kWgradVariants) {
      WgradBuild b2;
      if (build_bwd_filter_impl(d, nullptr, nullptr, nullptr, nullptr, di, b2, v[0], v[1]) == CONV2D_OK)
        need = std::max(need, b2.partial_bytes);
    }
    if (d.g > 1) {  // grouped: the one pass over the whole tensors (conv2d_bwd_filter_ex)
      Desc t = d;
      t.C = d.g * d.C;
      t.K = d.g * d.K;
      t.g = 1;
      WgradBuild w1;
      if (build_bwd_filter(t, nullptr, nullptr, nullptr, nullptr, di, w1) == CONV2D_OK) {
        need = std::max(need, w1.partial_bytes);
        for (const auto& v : kWgradVariants) {
          WgradBuild b2;
          if (build_bwd_filter_impl(t, nullptr, nullptr, nullptr, nullptr, di, b2, v[0], v[1]) == CONV2D_OK)
            need = std::max(need, b2.partial_bytes);
        }
      }
    }
    *bytes = std::max(phased, align_ws(need) + chan_sum_bytes(d));
    return CONV2D_OK;
  }
  return CONV2D_ERR_BAD_OP;
}
}  // namespace

extern "C" {


// Forward / backward-data: the plan (one or more tap passes) is made once per descriptor
// (cached with the group-0 addresses) and each group runs it with its own tensor slices:
// source, destination and bias channels of the group, the group's filter rows; the
// repacked filters reuse the workspace group after group (stream order).
static int run_tap(int op, const Desc& d, int groups, const void* src, const void* w, const void* bias, float beta,
                   int mode, void* dst, void* ws, size_t wsb, void* stream) {
  if (mode != CONV2D_MODE_CROSS_CORRELATION && mode != CONV2D_MODE_CONVOLUTION) return CONV2D_ERR_BAD_DESC;
  int rc = validate(d);
  if (rc) return rc;
  Desc dg;
  rc = group_desc(d, groups, dg);
  if (rc) return rc;
  rc = check_ptrs(src, w, dst, d.dt);
  if (rc) return rc;
  const DevInfo di = device_info();
  if (!di.ok) return CONV2D_ERR_DEVICE;
  if (bias != nullptr && ((uintptr_t)bias & (d.dt == CONV2D_DTYPE_F32 ? 3 : 1))) return CONV2D_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t esz = d.dt == CONV2D_DTYPE_F32 ? 4 : 2;
  const bool fwd = op == CONV2D_OP_FWD;
  // per-group element offsets of the source, destination, filter and bias slices
  const size_t src_g = fwd ? (size_t)dg.C * dg.H * dg.W : (size_t)dg.K * dg.P * dg.Q;
  const size_t dst_g = fwd ? (size_t)dg.K * dg.P * dg.Q : (size_t)dg.C * dg.H * dg.W;
  const size_t w_g = (size_t)dg.K * dg.C * dg.R * dg.S;
  const size_t bias_g = fwd ? (size_t)dg.K : (size_t)dg.C;
  if (is_depthwise(dg)) {  // direct kernels, every group in one launch, no workspace
    DwPlan dp = dw_plan(d, dg, di.sms);
    (fwd ? dp.x : dp.dy) = src;
    dp.w = w;
    dp.out = dst;
    dp.bias = bias;
    dp.beta = beta;
    dp.flip = mode == CONV2D_MODE_CONVOLUTION ? 1 : 0;
    return launch_err(fwd ? launch_dw_fwd(dp, d.dt, di.sms, st) : launch_dw_bwd_data(dp, d.dt, di.sms, st));
  }
  TapSet set;
  // Grouped layers: one pass over the whole tensors with the filter packed block-diagonally (zero
  // between channels of different groups) when that plans.  It costs the ungrouped op whatever
  // the group count (groups times the grouped multiply-adds, at the ungrouped tile width, one set
  // of packs, fills and epilogues); one pass per group costs groups times a pass whose tile is
  // only K/groups wide.  Measured on the ResNet 3x3 layer (ungrouped 30 us): one pass per group
  // 41 / 55 / 113 / 236 us forward at 2 / 4 / 8 / 16 groups, block-diagonal 29-30 us; the
  // deconvolution layer at 4 groups 69 -> 52 us forward, 69 -> 55 us backward-data (at 2 groups
  // 57 -> 52 forward, 55 -> 57 backward-data).
  bool blockdiag = false;
  if (blockdiag_groups(op, d, groups)) {
    const PlanKey bkey = make_key(op, d, src, w, dst, ws);
    blockdiag = g_tap_plans.get(bkey, set);
    if (!blockdiag && build_tap_set(op, d, src, w, dst, ws, di, set, true) == CONV2D_OK) {
      g_tap_plans.put(bkey, set);
      blockdiag = true;
    }
  }
  if (!fwd && !blockdiag) {  // few input channels: the scatter-form kernel (no workspace)
    C2iPlan cp;
    const PlanKey ckey = make_key(op, dg, nullptr, nullptr, nullptr, nullptr);
    bool have = g_c2i_plans.get(ckey, cp);
    if (!have && build_c2i(dg, src, w, dst, di, cp) == CONV2D_OK) {
      g_c2i_plans.put(ckey, cp);
      have = true;
    }
    if (have) {
      for (int gi = 0; gi < groups; ++gi) {
        cp.dy = byte_ptr(src) + gi * src_g * esz;
        cp.dx = const_cast<uint8_t*>(byte_ptr(dst)) + gi * dst_g * esz;
        cp.w = byte_ptr(w) + gi * w_g * esz;
        cp.bias = bias != nullptr ? byte_ptr(bias) + gi * bias_g * esz : nullptr;
        cp.beta = beta;
        cp.flip = mode == CONV2D_MODE_CONVOLUTION ? 1 : 0;
        cp.use_tma = cp.nraw_tma > 0 && encode_c2i_dy_map(&cp.tm_dy, cp.dy, cp) ? 1 : 0;
        cp.nraw = cp.use_tma ? cp.nraw_tma : 0;
        rc = launch_err(launch_c2i(cp, di.sms, st));
        if (rc) return rc;
      }
      return CONV2D_OK;
    }
  }
  if (!blockdiag) {
    const PlanKey key = make_key(op, dg, src, w, dst, ws);
    if (!g_tap_plans.get(key, set)) {
      rc = build_tap_set(op, dg, src, w, dst, ws, di, set, true);
      if (rc) return rc;
      g_tap_plans.put(key, set);
    }
  }
  rc = check_ws(ws, wsb, set.pack_bytes);
  if (rc) return rc;
  for (int gi = 0; gi < (blockdiag ? 1 : groups); ++gi)
    for (size_t pi = 0; pi < set.pass.size(); ++pi) {
      TapBuild& b = set.pass[pi];
      // per-call epilogue inputs and mode (not part of the cached plan); later passes add on
      b.p.beta = pi == 0 ? beta : 1.f;
      b.pp.flip = mode == CONV2D_MODE_CONVOLUTION ? 1 : 0;
      b.pp.C = dg.C;  // the filter's channels per group (K x C/groups x R x S)
      b.pp.gs = blockdiag ? (fwd ? dg.C : dg.K) : 0;
      b.pp.gd = blockdiag ? (fwd ? dg.K : dg.C) : 0;
      b.p.src = byte_ptr(src) + gi * src_g * esz;
      b.p.dst = const_cast<uint8_t*>(byte_ptr(dst)) + gi * dst_g * esz;
      b.pp.w = byte_ptr(w) + gi * w_g * esz;
      b.p.bias = bias != nullptr && pi == 0 ? byte_ptr(bias) + gi * bias_g * esz : nullptr;
      if (b.p.a_tma) {  // the group's source, packed channel-chunk-wise for the tensor copies
        b.px.src = b.p.src;
        if (b.pack_bytes) {  // with the filter pack in the same launch
          rc = launch_err(launch_tap_packs(b.px, b.pp, d.dt, di.sms, st));
        } else {
          NhwcPackPlan none;
          std::memset(&none, 0, sizeof(none));
          rc = launch_err(launch_nhwc_pack(b.px, none, d.dt, di.sms, st));
        }
        if (rc) return rc;
      } else if (b.pack_bytes) {
        rc = launch_err(launch_pack_filter(b.pp, d.dt, st));
        if (rc) return rc;
      }
      rc = launch_err(launch_tap_gemm(b.p, d.dt, b.grid, st));
      if (rc) return rc;
    }
  return CONV2D_OK;
}

int conv2d_fwd(int N, int C, int H, int W, int K, int R, int S, int pad_h, int pad_w, int stride_h,
               int stride_w, int P, int Q, int dtype, const void* x, const void* w, void* y, void* workspace,
               size_t workspace_bytes, void* stream) {
  const Desc d{N, C, H, W, K, R, S, pad_h, pad_w, stride_h, stride_w, P, Q, dtype};
  return run_tap(CONV2D_OP_FWD, d, 1, x, w, nullptr, 0.f, CONV2D_MODE_CROSS_CORRELATION, y, workspace,
                 workspace_bytes, stream);
}

int conv2d_fwd_ex(int N, int C, int H, int W, int K, int R, int S, int pad_h, int pad_w, int stride_h,
                  int stride_w, int P, int Q, int dil_h, int dil_w, int groups, int dtype, int mode, const void* x,
                  const void* w, const void* bias, float beta, void* y, void* workspace, size_t workspace_bytes,
                  void* stream) {
  const Desc d{N, C, H, W, K, R, S, pad_h, pad_w, stride_h, stride_w, P, Q, dtype, dil_h, dil_w};
  return run_tap(CONV2D_OP_FWD, d, groups, x, w, bias, beta, mode, y, workspace, workspace_bytes, stream);
}

int conv2d_bwd_data(int N, int C, int H, int W, int K, int R, int S, int pad_h, int pad_w, int stride_h,
                    int stride_w, int P, int Q, int dtype, const void* dy, const void* w, void* dx,
                    void* workspace, size_t workspace_bytes, void* stream) {
  const Desc d{N, C, H, W, K, R, S, pad_h, pad_w, stride_h, stride_w, P, Q, dtype};
  return run_tap(CONV2D_OP_BWD_DATA, d, 1, dy, w, nullptr, 0.f, CONV2D_MODE_CROSS_CORRELATION, dx, workspace,
                 workspace_bytes, stream);
}

int conv2d_bwd_data_ex(int N, int C, int H, int W, int K, int R, int S, int pad_h, int pad_w, int stride_h,
                       int stride_w, int P, int Q, int dil_h, int dil_w, int groups, int dtype, int mode,
                       const void* dy, const void* w, const void* bias, float beta, void* dx, void* workspace,
                       size_t workspace_bytes, void* stream) {
  const Desc d{N, C, H, W, K, R, S, pad_h, pad_w, stride_h, stride_w, P, Q, dtype, dil_h, dil_w};
  return run_tap(CONV2D_OP_BWD_DATA, d, groups, dy, w, bias, beta, mode, dx, workspace, workspace_bytes, stream);
}

int conv2d_bwd(int N, int C, int H, int W, int K, int R, int S, int pad_h, int pad_w, int stride_h, int stride_w,
               int P, int Q, int dtype, const void* x, const void* w, const void* dy, void* dx, void* dw,
               void* workspace, size_t workspace_bytes, void* stream) {
  const Desc d{N, C, H, W, K, R, S, pad_h, pad_w, stride_h, stride_w, P, Q, dtype};
  int rc = validate(d);
  if (rc) return rc;
  rc = check_ptrs(x, w, dy, dtype);
  if (rc) return rc;
  rc = check_ptrs(dx, dw, dy, dtype);
  if (rc) return rc;
  const DevInfo di = device_info();
  if (!di.ok) return CONV2D_ERR_DEVICE;
  FusedBwd f;
  const PlanKey key = make_key(kFusedKey, d, x, dy, dw, workspace);
  if (!g_fused_plans.get(key, f)) {
    rc = build_fused_bwd(d, x, w, dy, dx, dw, workspace, di, f);
    if (rc) return rc;
    if (workspace != nullptr) g_fused_plans.put(key, f);
  }
  if (!f.fused) {  // one op after the other, each planned on its own
    rc = conv2d_bwd_data(N, C, H, W, K, R, S, pad_h, pad_w, stride_h, stride_w, P, Q, dtype, dy, w, dx, workspace,
                         workspace_bytes, stream);
    if (rc) return rc;
    return conv2d_bwd_filter(N, C, H, W, K, R, S, pad_h, pad_w, stride_h, stride_w, P, Q, dtype, x, dy, dw,
                             workspace, workspace_bytes, stream);
  }
  rc = check_ws(workspace, workspace_bytes, f.need);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MnBuild& mb = f.mb;
  mb.px.src = x;
  mb.pd.src = dy;
  mb.rp.dw = dw;
  mb.rp.beta = 0.f;
  mb.rp.flip = 0;
  TapBuild& b = f.set.pass[0];
  b.p.src = dy;  // per call: the plan is cached under x, dy, dw and the workspace only
  b.p.dst = dx;
  b.pp.w = w;
  b.p.beta = 0.f;
  b.p.bias = nullptr;
  b.pp.flip = 0;
  // x and dy packed once; the backward-data GEMM (after its filter pack) reads the dy pack
  rc = launch_err(launch_nhwc_pack(mb.px, mb.pd, dtype, di.sms, st));
  if (rc) return rc;
  if (b.pack_bytes) {
    rc = launch_err(launch_pack_filter(b.pp, dtype, st));
    if (rc) return rc;
  }
  rc = launch_err(launch_tap_gemm(b.p, dtype, b.grid, st));
  if (rc) return rc;
  rc = launch_err(launch_wgrad_mn(mb.p, mb.grid, st));
  if (rc) return rc;
  return launch_err(launch_wgrad_reduce_t(mb.rp, dtype, di.sms, st));
}

int conv2d_bwd_filter(int N, int C, int H, int W, int K, int R, int S, int pad_h, int pad_w, int stride_h,
                      int stride_w, int P, int Q, int dtype, const void* x, const void* dy, void* dw,
                      void* workspace, size_t workspace_bytes, void* stream) {
  return conv2d_bwd_filter_ex(N, C, H, W, K, R, S, pad_h, pad_w, stride_h, stride_w, P, Q, 1, 1, 1, dtype,
                              CONV2D_MODE_CROSS_CORRELATION, x, dy, 0.f, dw, nullptr, nullptr, workspace,
                              workspace_bytes, stream);
}

int conv2d_bwd_filter_ex(int N, int C, int H, int W, int K, int R, int S, int pad_h, int pad_w, int stride_h,
                         int stride_w, int P, int Q, int dil_h, int dil_w, int groups, int dtype, int mode,
                         const void* x, const void* dy, float beta, void* dw, void* db_k, void* db_c, void* workspace,
                         size_t workspace_bytes, void* stream) {
  const Desc d{N, C, H, W, K, R, S, pad_h, pad_w, stride_h, stride_w, P, Q, dtype, dil_h, dil_w};
  if (mode != CONV2D_MODE_CROSS_CORRELATION && mode != CONV2D_MODE_CONVOLUTION) return CONV2D_ERR_BAD_DESC;
  int rc = validate(d);
  if (rc) return rc;
  Desc dg;
  rc = group_desc(d, groups, dg);
  if (rc) return rc;
  rc = check_ptrs(x, dy, dw, d.dt);
  if (rc) return rc;
  const uintptr_t am = d.dt == CONV2D_DTYPE_F32 ? 3 : 1;
  if (((uintptr_t)db_k & am) || ((uintptr_t)db_c & am)) return CONV2D_ERR_ALIGN;
  const DevInfo di = device_info();
  if (!di.ok) return CONV2D_ERR_DEVICE;
  const bool sums = db_k != nullptr || db_c != nullptr;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t esz = d.dt == CONV2D_DTYPE_F32 ? 4 : 2;
  size_t sum0 = 0;
  bool phases_run = false;
  // Depthwise: the direct partial sums over image ranges and their fixed-order reduce.
  if (is_depthwise(dg)) {
    DwPlan dp = dw_plan(d, dg, di.sms);
    dp.x = x;
    dp.dy = dy;
    dp.out = dw;
    dp.beta = beta;
    dp.flip = mode == CONV2D_MODE_CONVOLUTION ? 1 : 0;
    const size_t part = align_ws(dw_partial_bytes(dp));
    rc = check_ws(workspace, workspace_bytes, part + (sums ? chan_sum_bytes(d) : 0));
    if (rc) return rc;
    dp.partial = static_cast<float*>(workspace);
    rc = launch_err(launch_dw_bwd_filter(dp, d.dt, di.sms, st));
    if (rc) return rc;
    sum0 = part;
    phases_run = true;  // (the other paths below are skipped)
  }
  // bf16: x and dy packed into channel-chunked planes, then one tensor-copy-fed GEMM and the
  // fixed-order reduce.  One plan serves every group (its tensor maps address the workspace);
  // each group packs its own slices into the workspace in stream order.
  if (!phases_run && d.dt == CONV2D_DTYPE_BF16 && workspace != nullptr) {
    MnBuild mb;
    // Grouped: first the whole tensors in one pass (the full K x C gradient; the reduce keeps
    // the diagonal blocks), else one pass per group.
    bool whole = false;
    if (groups > 1) {
      const PlanKey wkey = make_key(kMnKey, d, nullptr, nullptr, nullptr, workspace);
      whole = g_mn_plans.get(wkey, mb);
      if (!whole && build_wgrad_mn(d, x, dy, dw, workspace, di, mb) == CONV2D_OK) {
        g_mn_plans.put(wkey, mb);
        whole = true;
      }
    }
    const PlanKey key = make_key(kMnKey, dg, nullptr, nullptr, nullptr, workspace);
    bool have = whole || g_mn_plans.get(key, mb);
    if (!have) {
      rc = build_wgrad_mn(dg, x, dy, dw, workspace, di, mb);
      if (rc == CONV2D_OK) {
        g_mn_plans.put(key, mb);
        have = true;
      } else if (rc != CONV2D_ERR_UNSUPPORTED) {
        return rc;
      }
    }
    if (have) {
      rc = check_ws(workspace, workspace_bytes, mn_ws_bytes(mb) + (sums ? chan_sum_bytes(d) : 0));
      if (rc) return rc;
      mb.rp.gk = whole ? dg.K : 0;
      mb.rp.gc = whole ? dg.C : 0;
      for (int gi = 0; gi < (whole ? 1 : groups); ++gi) {
        mb.px.src = byte_ptr(x) + gi * (size_t)dg.C * dg.H * dg.W * esz;
        mb.pd.src = byte_ptr(dy) + gi * (size_t)dg.K * dg.P * dg.Q * esz;
        mb.rp.dw = const_cast<uint8_t*>(byte_ptr(dw)) + gi * (size_t)dg.K * dg.C * dg.R * dg.S * esz;
        mb.rp.beta = beta;  // per-call (not part of the cached plan)
        mb.rp.flip = mode == CONV2D_MODE_CONVOLUTION ? 1 : 0;
        rc = launch_err(launch_nhwc_pack(mb.px, mb.pd, d.dt, di.sms, st));
        if (rc) return rc;
        rc = launch_err(launch_wgrad_mn(mb.p, mb.grid, st));
        if (rc) return rc;
        rc = launch_err(launch_wgrad_reduce_t(mb.rp, d.dt, di.sms, st));
        if (rc) return rc;
      }
      sum0 = mn_ws_bytes(mb);
      phases_run = true;  // (the other paths below are skipped)
    }
  }
  // Strided filters: x into stride-phase planes once, then one stride-1 pass per phase and
  // group (all planned before anything is enqueued; one problem if a phase has no plan).
  const PhaseLayout L = phase_layout(dg);
  if (!phases_run && L.on && workspace != nullptr && phase_need(dg, di) != 0) {
    uint8_t* wsp = static_cast<uint8_t*>(workspace);
    std::vector<std::vector<WgradBuild>> gp((size_t)groups);
    size_t partial = 0;
    bool phased = true;
    for (int gi = 0; gi < groups && phased; ++gi) {
      const void* dyg = byte_ptr(dy) + gi * (size_t)dg.K * dg.P * dg.Q * esz;
      void* dwg = const_cast<uint8_t*>(byte_ptr(dw)) + gi * (size_t)dg.K * dg.C * dg.R * dg.S * esz;
      rc = plan_phases(dg, L, wsp, dyg, dwg, wsp + L.xs_bytes, gi, di, gp[(size_t)gi]);
      if (rc == CONV2D_ERR_UNSUPPORTED) phased = false;
      else if (rc) return rc;
      for (const WgradBuild& wb : gp[(size_t)gi]) partial = std::max(partial, wb.partial_bytes);
    }
    if (phased) {
      // the phases must stage less than the problem as a whole (group 0's plan, cached under
      // the key the per-group loop below uses)
      WgradBuild whole;
      const PlanKey key = make_key(CONV2D_OP_BWD_FILTER, dg, x, dy, dw, workspace);
      bool have_whole = g_wgrad_plans.get(key, whole);
      if (!have_whole && build_bwd_filter(dg, x, dy, dw, workspace, di, whole) == CONV2D_OK) {
        g_wgrad_plans.put(key, whole);
        have_whole = true;
      }
      phased = phases_stage_less(gp[0], have_whole ? &whole.p : nullptr, d.dt);
    }
    if (phased) {
      rc = check_ws(workspace, workspace_bytes,
                    L.xs_bytes + (sums ? align_ws(partial) + chan_sum_bytes(d) : partial));
      if (rc) return rc;
      const S2dPlan sp{x, wsp, d.N, d.C, d.H, d.W, d.sh, d.sw, L.Hp, L.Wp};
      rc = launch_err(launch_space_to_depth(sp, d.dt, di.sms, st));
      if (rc) return rc;
      for (auto& phases : gp)
        for (WgradBuild& wb : phases) {
          wb.rp.beta = beta;  // per-call (not part of the cached plan)
          wb.rp.flip = mode == CONV2D_MODE_CONVOLUTION ? 1 : 0;
          rc = launch_err(launch_wgrad(wb.p, d.dt, wb.grid, st));
          if (rc) return rc;
          rc = launch_err(launch_wgrad_reduce(wb.rp, d.dt, di.sms, st));
          if (rc) return rc;
        }
      sum0 = L.xs_bytes + align_ws(partial);
      phases_run = true;
    }
  }
  // Grouped layers: one split-K pass over the whole tensors whose reduce keeps only the diagonal
  // blocks of the full K x C gradient (the ungrouped op's cost whatever the group count, against
  // groups passes whose GEMMs are only K/groups wide).
  if (!phases_run && groups > 1) {
    WgradBuild b;
    const PlanKey key = make_key(CONV2D_OP_BWD_FILTER, d, x, dy, dw, workspace);
    bool have = g_wgrad_plans.get(key, b);
    if (!have && build_bwd_filter(d, x, dy, dw, workspace, di, b) == CONV2D_OK) {
      g_wgrad_plans.put(key, b);
      have = true;
    }
    if (have) {
      rc = check_ws(workspace, workspace_bytes, sums ? align_ws(b.partial_bytes) + chan_sum_bytes(d) : b.partial_bytes);
      if (rc) return rc;
      b.rp.beta = beta;  // per-call (not part of the cached plan)
      b.rp.flip = mode == CONV2D_MODE_CONVOLUTION ? 1 : 0;
      b.rp.gk = dg.K;
      b.rp.gc = dg.C;
      rc = launch_err(launch_wgrad(b.p, d.dt, b.grid, st));
      if (rc) return rc;
      rc = launch_err(launch_wgrad_reduce(b.rp, d.dt, di.sms, st));
      if (rc) return rc;
      sum0 = align_ws(b.partial_bytes);
      phases_run = true;
    }
  }
  // One split-K pass per group on the group's slices (x channels, dy channels, dw rows);
  // the split partials reuse the workspace group after group (stream order).  The plans
  // embed the slices' addresses (tensor maps), so each group has its own cached plan.
  for (int gi = 0; gi < groups && !phases_run; ++gi) {
    const void* xg = byte_ptr(x) + gi * (size_t)dg.C * dg.H * dg.W * esz;
    const void* dyg = byte_ptr(dy) + gi * (size_t)dg.K * dg.P * dg.Q * esz;
    void* dwg = const_cast<uint8_t*>(byte_ptr(dw)) + gi * (size_t)dg.K * dg.C * dg.R * dg.S * esz;
    WgradBuild b;
    const PlanKey key = make_key(CONV2D_OP_BWD_FILTER, dg, xg, dyg, dwg, workspace);
    if (!g_wgrad_plans.get(key, b)) {
      rc = build_bwd_filter(dg, xg, dyg, dwg, workspace, di, b);
      if (rc) return rc;
      g_wgrad_plans.put(key, b);
    }
    sum0 = std::max(sum0, align_ws(b.partial_bytes));
    rc = check_ws(workspace, workspace_bytes, sums ? align_ws(b.partial_bytes) + chan_sum_bytes(d) : b.partial_bytes);
    if (rc) return rc;
    b.rp.beta = beta;  // per-call (not part of the cached plan)
    b.rp.flip = mode == CONV2D_MODE_CONVOLUTION ? 1 : 0;
    rc = launch_err(launch_wgrad(b.p, d.dt, b.grid, st));
    if (rc) return rc;
    rc = launch_err(launch_wgrad_reduce(b.rp, d.dt, di.sms, st));
    if (rc) return rc;
  }
  // Bias gradients, both in one launch pair: the conv bias gradient db_k sums dy over images
  // and output pixels per output channel k; the deconvolution bias gradient db_c sums x (the
  // deconvolution's output gradient) over images and pixels per channel c.
  uint8_t* wsb = static_cast<uint8_t*>(workspace) + sum0;
  ChanSumPlan sk{}, sc{};
  if (db_k != nullptr) {
    sk = ChanSumPlan{dy, db_k, reinterpret_cast<float*>(wsb), d.N, d.K, (long long)d.P * d.Q, beta, 0, 0};
    chan_sum_blocks(sk, d.dt);
  }
  if (db_c != nullptr) {
    sc = ChanSumPlan{x, db_c, reinterpret_cast<float*>(wsb + align_ws((size_t)d.K * d.N * sizeof(float))), d.N, d.C,
                     (long long)d.H * d.W, beta, 0, 0};
    chan_sum_blocks(sc, d.dt);
  }
  if (sums) {
    rc = launch_err(launch_chan_sum(db_k != nullptr ? sk : sc, db_k != nullptr ? sc : ChanSumPlan{}, d.dt, st), 2);
    if (rc) return rc;
  }
  return CONV2D_OK;
}

int conv2d_fwd_noalloc(int N, int C, int H, int W, int K, int R, int S, int pad_h, int pad_w, int stride_h,
                       int stride_w, int P, int Q, int dtype, const void* x, const void* w, void* y,
                       void* stream) {
  const Desc d{N, C, H, W, K, R, S, pad_h, pad_w, stride_h, stride_w, P, Q, dtype};
  int rc = validate(d);
  if (rc) return rc;
  rc = check_ptrs(x, w, y, d.dt);
  if (rc) return rc;
  const DevInfo di = device_info();
  if (!di.ok) return CONV2D_ERR_DEVICE;
  void* scratch = nullptr;
  if (noalloc_scratch_ptr(&scratch) != cudaSuccess) {
    cudaGetLastError();
    return CONV2D_ERR_DEVICE;
  }
  // The plan conv2d_fwd makes (one or more tap passes), with the scratch as its workspace.
  TapSet set;
  const PlanKey key = make_key(CONV2D_OP_FWD, d, x, w, y, scratch);
  if (!g_tap_plans.get(key, set)) {
    rc = build_tap_set(CONV2D_OP_FWD, d, x, w, y, scratch, di, set, false);
    if (rc) return rc;
    g_tap_plans.put(key, set);
  }
  if (set.pack_bytes > noalloc_scratch_capacity()) return CONV2D_ERR_NOALLOC_LIMIT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (size_t pi = 0; pi < set.pass.size(); ++pi) {
    TapBuild& b = set.pass[pi];
    b.p.beta = pi == 0 ? 0.f : 1.f;  // later passes add onto the output the first one wrote
    b.p.bias = nullptr;
    b.pp.flip = 0;
    if (b.pack_bytes) {
      rc = launch_err(launch_pack_filter(b.pp, d.dt, st));
      if (rc) return rc;
    }
    rc = launch_err(launch_tap_gemm(b.p, d.dt, b.grid, st));
    if (rc) return rc;
  }
  return CONV2D_OK;
}

unsigned long long conv2d_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int conv2d_device_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return CONV2D_ERR_LAUNCH;
  }
  const int a = tap_gemm_take_error();
  const int b = wgrad_take_error();
  const int c = wgrad_mn_take_error();
  const int e = c2i_take_error();
  if (a < 0 || b < 0 || c < 0 || e < 0) return CONV2D_ERR_LAUNCH;
  if (a == DEV_ERR_LAYOUT || b == DEV_ERR_LAYOUT || c == DEV_ERR_LAYOUT || e == DEV_ERR_LAYOUT)
    return CONV2D_ERR_LAUNCH;
  if (a || b || c || e) return CONV2D_ERR_DEVICE_TIMEOUT;
  return CONV2D_OK;
}

const char* conv2d_strerror(int code) {
  switch (code) {
    case CONV2D_OK: return "success";
    case CONV2D_ERR_BAD_DESC: return "bad descriptor: a dimension <= 0, pad < 0 or stride < 1";
    case CONV2D_ERR_SHAPE: return "P/Q differ from floor((H+2*pad-R)/stride)+1, or are < 1";
    case CONV2D_ERR_NULLPTR: return "NULL tensor or workspace pointer";
    case CONV2D_ERR_ALIGN: return "misaligned pointer";
    case CONV2D_ERR_DTYPE: return "unknown dtype";
    case CONV2D_ERR_WORKSPACE: return "workspace smaller than conv2d_workspace_size()";
    case CONV2D_ERR_TOO_LARGE: return "a tensor has 2^31 or more elements";
    case CONV2D_ERR_LAUNCH: return "CUDA launch or stream error";
    case CONV2D_ERR_DEVICE: return "no sm_100-family CUDA device is current";
    case CONV2D_ERR_DEVICE_TIMEOUT: return "a kernel's bounded pipeline wait expired";
    case CONV2D_ERR_UNSUPPORTED: return "unsupported geometry (R*S > 256, stride_h*stride_w > 16, or no tile fits in shared memory)";
    case CONV2D_ERR_BAD_OP: return "unknown op";
    case CONV2D_ERR_NOALLOC_LIMIT:
      return "conv2d_fwd_noalloc: the packed filter exceeds the library's fixed 8 MiB scratch";
    default: return "unknown error code";
  }
}

}  // extern "C"

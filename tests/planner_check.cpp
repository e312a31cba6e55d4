// Host-only check of the launch planner (no GPU): plans the three ops for a list of shapes
// and verifies the invariants the kernels rely on -- shared-memory and TMEM budgets, staged
// rows covering every tap offset, every forward / backward-data tap reading the pixel the
// definition names (also across the passes of large filters), ring sizes covering the
// positions in flight, bank-spread ring pitches, and that every (channel, tap) of the
// filter gradient is produced exactly once.
// Tensor maps are not encoded (a stand-in encoder accepts every map), so the copy-engine
// plans are checked as they would be planned for aligned tensors.  Prints one line per
// violation and exits with the number of violations (capped at 100).
#include <cuda.h>
#include <cuda_runtime.h>

static CUresult accept_map(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*, const cuuint64_t*,
                           const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                           CUtensorMapL2promotion, CUtensorMapFloatOOBfill) {
  return CUDA_SUCCESS;
}
static cudaError_t entry_point_stand_in(const char*, void** f, unsigned int, unsigned long long,
                                        cudaDriverEntryPointQueryResult* q) {
  *f = (void*)&accept_map;
  *q = cudaDriverEntryPointSuccess;
  return cudaSuccess;
}
#define cudaGetDriverEntryPointByVersion entry_point_stand_in
#include "conv2d_api.cpp"

#include <cstdio>
#include <vector>

namespace {

int g_fail = 0;

void fail(const char* nm, const char* op, const char* what) {
  ++g_fail;
  std::printf("FAIL %s %s: %s\n", nm, op, what);
}

struct Shape {
  const char* nm;
  int N, C, H, W, K, R, S, ph, pw, sh, sw, dt;
  int dh, dw, g;
  int passes[2];  // tap passes expected for forward and backward-data
};

void check_tap(const char* nm, const char* op, const TapBuild& b, const DevInfo& di) {
  const TapPlan& p = b.p;
  if (tap_gemm_smem_bytes(p) > di.smem_optin) fail(nm, op, "shared memory over budget");
  if (p.tmem_cols > 512 || p.ACCB * p.MH * p.NT > p.tmem_cols) fail(nm, op, "TMEM over budget");
  if (p.rows < 128 * p.MH) fail(nm, op, "staged rows below the tile height");
  for (int ph = 0; ph < p.nph; ++ph)
    for (int t = p.ph_tap_begin[ph]; t < p.ph_tap_begin[ph] + p.ph_ntaps[ph]; ++t)
      if (p.tap_off[t] < 0 || p.tap_off[t] + 128 * p.MH > p.rows) fail(nm, op, "tap offset beyond the staged rows");
  if (p.NT % 16 || p.NT > 256 || (p.MH != 1 && p.MH != 2)) fail(nm, op, "tile shape");
  if (p.Mtot >= (1ll << 31)) fail(nm, op, "position space too large");
}

// Every real tap of every pass reads, for every output the plan writes, the source pixel the
// definition names: forward (p*sh - ph + r*dh, q*sw - pw + s*dw) of x; backward-data
// ((h + ph - r*dh) / sh, (w + pw - s*dw) / sw) of dy.  The kernel's read follows the linear
// space: the output at linear (e, f) reads linear position e*WL + f + tap offset of the tap's
// plane, whose pixel is (row * step + plane offset) in each dim; outputs outside the
// destination are not written, so their reads do not matter.  Every (r, s) must be a real
// tap of exactly one pass.
void check_tap_semantics(const char* nm, const char* op, const Desc& d, const TapSet& set, bool fwd) {
  std::vector<int> seen((size_t)d.R * d.S, 0);
  bool bad = false;
  for (const TapBuild& b : set.pass) {
    const TapPlan& p = b.p;
    for (int ph = 0; ph < p.nph && !bad; ++ph)
      for (int t = p.ph_tap_begin[ph]; t < p.ph_tap_begin[ph] + p.ph_ntaps[ph] && !bad; ++t) {
        const int r = b.pp.tap_r[t], s = b.pp.tap_s[t];
        if (r < 0) continue;  // zero-weight tap that pads a phase to an even count
        ++seen[(size_t)r * d.S + s];
        const int pl = p.tap_plane[t];
        for (int e = 0; e < p.EL && !bad; ++e)
          for (int f = 0; f < p.WL; ++f) {
            const int oh = e * p.ph_step_h + p.ph_off_h[ph], ow = f * p.ph_step_w + p.ph_off_w[ph];
            if (oh < 0 || oh >= p.Hd || ow < 0 || ow >= p.Wd) continue;  // not an output
            const long long L = (long long)e * p.WL + f + p.tap_off[t];
            const long long es = L / p.WL, fs = L % p.WL;
            if (es >= p.EL) {  // the kernel would read the next image's rows
              fail(nm, op, "a tap reads past its image in the linear space");
              bad = true;
              break;
            }
            const long long kh = es * p.pl_step_h + p.pl_off_h[pl], kw = fs * p.pl_step_w + p.pl_off_w[pl];
            long long dh, dwc;
            if (fwd) {
              dh = (long long)oh * d.sh - d.ph + r * d.dh;
              dwc = (long long)ow * d.sw - d.pw + s * d.dw;
            } else {
              const int nh = oh + d.ph - r * d.dh, nw = ow + d.pw - s * d.dw;
              if (((nh % d.sh) + d.sh) % d.sh != 0 || ((nw % d.sw) + d.sw) % d.sw != 0) {
                fail(nm, op, "a tap sits in a phase whose outputs it does not reach");
                bad = true;
                break;
              }
              dh = floor_div(nh, d.sh);
              dwc = floor_div(nw, d.sw);
            }
            if (kh != dh || kw != dwc) {
              fail(nm, op, fwd ? "a tap reads the wrong source pixel" : "a tap reads the wrong dy pixel");
              bad = true;
              break;
            }
          }
      }
  }
  for (size_t i = 0; i < seen.size(); ++i)
    if (seen[i] != 1) {
      fail(nm, op, "a filter tap is not in exactly one pass");
      break;
    }
}

void check_wgrad(const char* nm, const Desc& d, const WgradBuild& b, const DevInfo& di) {
  const char* op = "bwd_filter";
  const WgradPlan& p = b.p;
  // Every tap pairs dy at each output (e, f) with the x pixel the definition names
  // (e*sh - ph + r*dh, f*sw - pw + s*dw): x is read at linear e*WL + f + tap offset of the
  // tap's plane, without leaving the image; row-tap sharing shifts dy by j * tru_step rows
  // for filter row r0 + j, which needs offset(r0 + j) - offset(r0) = j * tru_step * WL.
  // (1x1 problems are planned on their flattened descriptor, one row of H*W pixels.)
  const Desc dd = flatten_pointwise(d);
  for (int r = 0; r < d.R; ++r)
    for (int s2 = 0; s2 < d.S; ++s2) {
      const int t = r * d.S + s2, pl = p.tap_plane[t];
      bool bad = false;
      for (int e = 0; e < dd.P && !bad; ++e)
        for (int f = 0; f < dd.Q; ++f) {
          const long long L = (long long)e * p.WL + f + p.tap_off[t];
          const long long es = L / p.WL, fs = L % p.WL;
          if (es >= p.EL || es * p.pl_step_h + p.pl_off_h[pl] != (long long)e * dd.sh - dd.ph + r * dd.dh ||
              fs * p.pl_step_w + p.pl_off_w[pl] != (long long)f * dd.sw - dd.pw + s2 * dd.dw) {
            fail(nm, op, "a tap pairs dy with the wrong x pixel");
            bad = true;
            break;
          }
        }
      if (p.TRU > 1 && r > 0 && p.tap_off[t] - p.tap_off[t - d.S] != p.tru_step * p.WL)
        fail(nm, op, "row-tap sharing: consecutive filter rows are not tru_step linear rows apart");
    }
  if (wgrad_smem_bytes(p, d.dt) > di.smem_optin) fail(nm, op, "shared memory over budget");
  if (128 + p.accb * p.G * p.TRU * p.NK > p.tmem_cols || p.tmem_cols > 512) fail(nm, op, "TMEM over budget");
  if (p.use_tma != 1 && p.rlen < p.stages * p.KB + p.max_off + 4) fail(nm, op, "slot ring shorter than the positions in flight");
  if (p.use_tma == 1) {
    // rows touched by the stages in flight: at most floor((S*KB + max_off - 1) / WL) + 2
    if ((long long)(p.NR - 2) * p.WL < (long long)p.stages * p.KB + p.max_off - 1) fail(nm, op, "x row ring too small");
    if (d.dt == 0 && p.WLx % 8 != 4) fail(nm, op, "x row pitch not 16 bytes past a multiple of 32");
    if (d.dt == 1 && p.WLx % 16 != 8) fail(nm, op, "x row pitch not 16 bytes past a multiple of 32");
  }
  if (p.TRU > 1) {
    if ((long long)(p.NRd - 1 - (p.TRU - 1) * p.tru_step) * p.WL <= (long long)p.stages * p.KB - 1)
      fail(nm, op, "dy row ring too small");
    if (p.WL % (d.dt == 0 ? 8 : 16)) fail(nm, op, "row width splits an MMA's chunk pair");
    if (p.use_tma != 1 || p.TPU != 1) fail(nm, op, "row-tap sharing outside the row ring");
  }
  if (p.KB % (d.dt == 0 ? 32 : 64)) fail(nm, op, "stage not a whole number of A buffers");
  // every row of every m-tile lies in the staged channels of its group, and every
  // (channel, tap) is produced exactly once
  std::vector<int> seen((size_t)d.C * p.RS, 0);
  for (int mg = 0; mg < p.n_mgroups; ++mg) {
    const int mt0 = mg * p.G;
    const int c_lo = ((4 * mt0) / p.upc) * p.Cg;
    for (int mt = mt0; mt < std::min(p.n_mtiles, mt0 + p.G); ++mt)
      for (int q = 0; q < 4; ++q)
        for (int l = 0; l < 32; ++l) {
          const int u = 4 * mt + q;
          if (u >= p.nunits) continue;
          const int cg = u / p.upc, tu = u % p.upc;
          int c, tap;
          bool v;
          if (p.TPU == 1) {
            c = cg * p.Cg + l;
            tap = p.unit_tap[tu];
            v = c < d.C;
          } else {
            const int tl = l / p.Cg;
            c = l - tl * p.Cg;
            tap = tu * p.TPU + tl;
            v = tl < p.TPU && tap < p.RS;
          }
          if (!v) continue;
          if (c - c_lo < 0 || c - c_lo >= p.xch) fail(nm, op, "row outside the group's staged channels");
          if (p.use_tma == 1 && c - c_lo >= p.xr) fail(nm, op, "row outside the row ring's channels");
          for (int j = 0; j < p.TRU; ++j) {
            if (tap / d.S + j >= d.R) break;
            ++seen[(size_t)c * p.RS + tap + j * d.S];
          }
        }
  }
  for (size_t i = 0; i < seen.size(); ++i)
    if (seen[i] != 1) {
      fail(nm, op, "a (channel, tap) of the filter gradient is not produced exactly once");
      break;
    }
}

// Strided backward-filter as stride phases: each phase plans and meets the invariants
// above; each of its taps reads, through the planes, the input pixel the definition names
// for every output; the placed taps cover the filter once.
void check_phases(const char* nm, const Desc& dg, const DevInfo& di, int& plans) {
  const PhaseLayout L = phase_layout(dg);
  if (!L.on) return;
  std::vector<WgradBuild> ph;
  void* xs = (void*)0x500000;
  if (plan_phases(dg, L, xs, (void*)0x300000, (void*)0x200000, (void*)0x600000, 0, di, ph) != CONV2D_OK) {
    fail(nm, "bwd_filter", "a stride phase has no plan");
    return;
  }
  std::vector<int> seen((size_t)dg.R * dg.S, 0);
  size_t i = 0;
  for (const StridePhase& a : L.rows)
    for (const StridePhase& b : L.cols) {
      const Desc q = phase_desc(dg, L, a, b);
      const WgradBuild& wb = ph[i++];
      check_wgrad(nm, q, wb, di);
      ++plans;
      // the plan addresses the caller's dy and the planes buffer with their real image strides
      if (wb.p.dy_nstride != (long long)dg.g * dg.K * dg.P * dg.Q)
        fail(nm, "bwd_filter", "phase plan's dy image stride differs from the dy tensor's");
      if (wb.p.x_nstride != (long long)dg.sh * dg.sw * dg.g * dg.C * L.Hp * L.Wp)
        fail(nm, "bwd_filter", "phase plan's x image stride differs from the planes buffer's");
      for (int r2 = 0; r2 < q.R; ++r2)
        for (int s2 = 0; s2 < q.S; ++s2) {
          const int r = wb.rp.r0 + wb.rp.rstep * r2, s = wb.rp.s0 + wb.rp.sstep * s2;
          if (r < 0 || r >= dg.R || s < 0 || s >= dg.S) {
            fail(nm, "bwd_filter", "a phase tap lies outside the filter");
            continue;
          }
          ++seen[(size_t)r * dg.S + s];
          for (int p = 0; p < dg.P; ++p)
            if (dg.sh * (p - q.ph + r2) + a.rho != p * dg.sh - dg.ph + r) fail(nm, "bwd_filter", "phase row");
          for (int qq = 0; qq < dg.Q; ++qq)
            if (dg.sw * (qq - q.pw + s2) + b.rho != qq * dg.sw - dg.pw + s) fail(nm, "bwd_filter", "phase column");
        }
      if (q.ph < 0 || q.pw < 0) fail(nm, "bwd_filter", "negative phase pad");
    }
  for (size_t t = 0; t < seen.size(); ++t)
    if (seen[t] != 1) {
      fail(nm, "bwd_filter", "a filter tap is not in exactly one stride phase");
      break;
    }
}

// The stride-phase choice on the strided workloads: the phases pay where x staging dominates
// (128 and 256 channels), not on the 3-channel stem, as measured.
void check_phase_choice(int& plans) {
  struct W { const char* nm; int v[12]; bool phases; } ws[] = {
      {"strided", {64, 128, 56, 56, 256, 3, 3, 1, 1, 2, 2, 0}, true},
      {"stem7x7", {64, 3, 224, 224, 64, 7, 7, 3, 3, 2, 2, 0}, false},
      {"deconv", {32, 256, 32, 32, 512, 4, 4, 1, 1, 2, 2, 1}, true},
  };
  DevInfo di;
  di.sms = 152;
  di.smem_optin = 232448;
  di.ok = true;
  for (const W& w : ws) {
    Desc d{};
    const int* v = w.v;
    d.N = v[0]; d.C = v[1]; d.H = v[2]; d.W = v[3]; d.K = v[4]; d.R = v[5]; d.S = v[6];
    d.ph = v[7]; d.pw = v[8]; d.sh = v[9]; d.sw = v[10]; d.dt = v[11];
    d.P = out_dim(d.H, d.ph, d.R, d.sh);
    d.Q = out_dim(d.W, d.pw, d.S, d.sw);
    const PhaseLayout L = phase_layout(d);
    std::vector<WgradBuild> ph;
    WgradBuild whole;
    if (plan_phases(d, L, (void*)0x500000, (void*)0x300000, (void*)0x200000, (void*)0x600000, 0, di, ph) != CONV2D_OK ||
        build_bwd_filter(d, (void*)0x100000, (void*)0x300000, (void*)0x200000, (void*)0x600000, di, whole) != CONV2D_OK) {
      fail(w.nm, "bwd_filter", "no plan");
      continue;
    }
    plans += 1 + (int)ph.size();
    if (phases_stage_less(ph, &whole.p, d.dt) != w.phases) fail(w.nm, "bwd_filter", "unexpected stride-phase choice");
    const size_t need = phase_need(d, di);
    if (need == 0 || need > kWorkspaceCap || need < L.xs_bytes) fail(w.nm, "bwd_filter", "stride-phase workspace");
  }
  // a layer whose x alone passes the workspace cap runs as a whole
  Desc big{};
  big.N = 112; big.C = 256; big.H = 96; big.W = 96; big.K = 256; big.R = 3; big.S = 3;
  big.ph = 1; big.pw = 1; big.sh = 2; big.sw = 2; big.dt = 0; big.P = 48; big.Q = 48;
  if (phase_need(big, di) != 0) fail("x_over_cap", "bwd_filter", "stride phases past the workspace cap");
}

}  // namespace

int main() {
  using namespace cg3;
  // The last field gives the tap passes expected for forward and backward-data.  The tap GEMM
  // stages the filter slices of every tap of a phase for each k-block; with a stride-1 15x15
  // filter and more than 4 fp32 (8 bf16) source channels that is 225 taps x 2 chunks x 16
  // columns x 16 bytes = 115 KB a stage, so two stages do not fit in shared memory and the
  // taps are split over passes.  With at most 4 (8) source channels two taps share one MMA
  // and the slices halve.  The source channels are C forward and K backward-data.
  std::vector<Shape> shapes = {
      {"tiny", 2, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1, 0, 1, 1, 1, {1, 1}},
      {"resnet3x3", 32, 64, 56, 56, 64, 3, 3, 1, 1, 1, 1, 0, 1, 1, 1, {1, 1}},
      {"resnet3x3_bf16", 32, 64, 56, 56, 64, 3, 3, 1, 1, 1, 1, 1, 1, 1, 1, {1, 1}},
      {"strided", 64, 128, 56, 56, 256, 3, 3, 1, 1, 2, 2, 0, 1, 1, 1, {1, 1}},
      {"pointwise", 128, 256, 14, 14, 1024, 1, 1, 0, 0, 1, 1, 0, 1, 1, 1, {1, 1}},
      {"stem7x7", 64, 3, 224, 224, 64, 7, 7, 3, 3, 2, 2, 0, 1, 1, 1, {1, 1}},
      {"deconv", 32, 256, 32, 32, 512, 4, 4, 1, 1, 2, 2, 1, 1, 1, 1, {1, 1}},
      {"c33", 3, 33, 9, 11, 40, 3, 3, 1, 1, 1, 1, 0, 1, 1, 1, {1, 1}},
      {"k300", 1, 17, 6, 6, 300, 3, 3, 1, 1, 1, 1, 0, 1, 1, 1, {1, 1}},
      {"c300", 2, 300, 5, 5, 20, 3, 3, 1, 1, 1, 1, 1, 1, 1, 1, {1, 1}},
      {"c5k300", 2, 5, 17, 13, 300, 5, 3, 2, 1, 2, 1, 1, 1, 1, 1, {1, 1}},
      {"r15", 1, 4, 40, 40, 8, 15, 15, 7, 7, 1, 1, 0, 1, 1, 1, {1, 2}},
      {"r15_k4", 1, 8, 40, 40, 4, 15, 15, 7, 7, 1, 1, 0, 1, 1, 1, {2, 1}},
      {"r16_c16", 1, 16, 40, 40, 16, 16, 16, 7, 7, 1, 1, 0, 1, 1, 1, {2, 2}},
      {"r16_s2_bf16", 2, 24, 40, 40, 20, 16, 16, 7, 7, 2, 2, 1, 1, 1, 1, {4, 1}},
      {"r1_s256", 1, 16, 4, 300, 16, 1, 256, 0, 3, 1, 1, 0, 1, 1, 1, {2, 2}},
      {"s32", 2, 40, 23, 19, 24, 3, 3, 1, 1, 3, 2, 1, 1, 1, 1, {1, 1}},
      {"hr", 1, 2, 6, 13, 2, 6, 13, 0, 0, 1, 1, 0, 1, 1, 1, {1, 1}},
      {"rows5", 1, 40, 16, 16, 48, 5, 3, 2, 1, 1, 1, 0, 1, 1, 1, {1, 1}},
      {"rows5_bf16", 1, 40, 16, 16, 48, 5, 3, 2, 1, 1, 1, 1, 1, 1, 1, {1, 1}},
      {"wide_k", 1, 32, 8, 8, 150, 3, 3, 1, 1, 1, 1, 0, 1, 1, 1, {1, 1}},
      {"wide_k_bf16", 1, 32, 8, 8, 150, 3, 3, 1, 1, 1, 1, 1, 1, 1, 1, {1, 1}},
      {"rect", 2, 48, 10, 16, 20, 3, 5, 1, 2, 1, 1, 0, 1, 1, 1, {1, 1}},
      {"big7", 8, 64, 32, 32, 64, 7, 7, 3, 3, 1, 1, 0, 1, 1, 1, {1, 1}},
      {"dil2", 2, 64, 16, 16, 64, 3, 3, 2, 2, 1, 1, 0, 2, 2, 1, {1, 1}},
      {"dil2_bf16", 2, 64, 16, 16, 64, 3, 3, 2, 2, 1, 1, 1, 2, 2, 1, {1, 1}},
      {"dil23", 1, 5, 20, 17, 7, 3, 2, 2, 1, 2, 1, 1, 2, 3, 1, {1, 1}},
      {"dil32", 1, 33, 15, 16, 40, 2, 3, 1, 2, 1, 2, 0, 3, 2, 1, {1, 1}},
      {"dil3_s2", 2, 3, 21, 21, 16, 3, 3, 3, 3, 2, 2, 1, 3, 3, 1, {1, 1}},
      {"grp3", 2, 6, 9, 10, 9, 3, 3, 1, 1, 1, 1, 0, 1, 1, 3, {1, 1}},
      {"grp2", 2, 64, 16, 16, 64, 3, 3, 1, 1, 1, 1, 0, 1, 1, 2, {1, 1}},
      {"depthwise", 1, 16, 12, 12, 16, 3, 3, 1, 1, 1, 1, 1, 1, 1, 16, {1, 1}},
      {"grp_dil", 2, 8, 13, 11, 6, 3, 3, 2, 2, 1, 2, 0, 2, 1, 2, {1, 1}},
      {"s3_r2", 1, 1, 7, 7, 1, 2, 2, 0, 0, 3, 3, 0, 1, 1, 1, {1, 1}},
      {"s2_9x9", 2, 3, 9, 9, 4, 3, 3, 1, 1, 2, 2, 0, 1, 1, 1, {1, 1}},
      {"s2_grp", 2, 8, 14, 13, 6, 3, 3, 1, 1, 2, 2, 1, 1, 1, 2, {1, 1}},
      {"s32_r5", 1, 40, 20, 19, 24, 5, 3, 2, 0, 2, 3, 0, 1, 1, 1, {1, 1}},
  };
  DevInfo di;
  di.sms = 152;
  di.smem_optin = 232448;
  di.ok = true;
  int plans = 0;
  for (const Shape& s : shapes) {
    Desc t{};
    t.N = s.N; t.C = s.C; t.H = s.H; t.W = s.W; t.K = s.K; t.R = s.R; t.S = s.S;
    t.ph = s.ph; t.pw = s.pw; t.sh = s.sh; t.sw = s.sw; t.dt = s.dt; t.dh = s.dh; t.dw = s.dw;
    t.P = out_dim(t.H, t.ph, t.dh * (t.R - 1) + 1, t.sh);
    t.Q = out_dim(t.W, t.pw, t.dw * (t.S - 1) + 1, t.sw);
    if (validate(t) != CONV2D_OK) { fail(s.nm, "desc", "descriptor rejected"); continue; }
    Desc d;
    if (group_desc(t, s.g, d) != CONV2D_OK) { fail(s.nm, "desc", "groups rejected"); continue; }
    void* px = (void*)0x100000;  // 16-byte aligned stand-in addresses
    void* pw = (void*)0x200000;
    void* py = (void*)0x300000;
    void* ws = (void*)0x400000;
    for (int op = 0; op < 2; ++op) {
      const char* opn = op == 0 ? "fwd" : "bwd_data";
      TapSet set;
      const int rc = op == 0 ? build_tap_set(CONV2D_OP_FWD, d, px, pw, py, ws, di, set)
                             : build_tap_set(CONV2D_OP_BWD_DATA, d, py, pw, px, ws, di, set);
      if (rc != CONV2D_OK) {
        fail(s.nm, opn, "no plan");
        continue;
      }
      if ((int)set.pass.size() != s.passes[op]) {
        std::printf("  %s %s: %d passes\n", s.nm, opn, (int)set.pass.size());
        fail(s.nm, opn, "unexpected number of tap passes");
      }
      for (const TapBuild& b : set.pass) {
        check_tap(s.nm, opn, b, di);
        ++plans;
      }
      check_tap_semantics(s.nm, opn, d, set, op == 0);
    }
    for (const auto& v : kWgradVariants) {  // every staging variant the planner may fall back to
      WgradBuild bw;
      const int rc = build_bwd_filter_impl(d, px, py, pw, ws, di, bw, v[0], v[1]);
      if (rc == CONV2D_ERR_UNSUPPORTED) continue;
      if (rc != CONV2D_OK) { fail(s.nm, "bwd_filter", "planner error"); continue; }
      check_wgrad(s.nm, d, bw, di);
      ++plans;
    }
    WgradBuild bw;
    if (build_bwd_filter(d, px, py, pw, ws, di, bw) != CONV2D_OK) fail(s.nm, "bwd_filter", "no plan");
    check_phases(s.nm, d, di, plans);
  }
  check_phase_choice(plans);
  int refused = 0;  // backward-filter problems refused with CONV2D_ERR_UNSUPPORTED
  // seeded random descriptors: every op plans (or is refused as documented) and meets the
  // same invariants and definition checks
  {
    unsigned long long st = 0x9E3779B97F4A7C15ull;
    auto rnd = [&](int lo, int hi) {  // inclusive, splitmix64
      st += 0x9E3779B97F4A7C15ull;
      unsigned long long z = st;
      z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
      z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
      z ^= z >> 31;
      return lo + (int)(z % (unsigned long long)(hi - lo + 1));
    };
    int drawn = 0;
    while (drawn < 550) {
      // 400 small descriptors, then 150 at layer scale (large images and channel counts)
      const bool big = drawn >= 400;
      Desc t{};
      t.N = big ? rnd(1, 64) : rnd(1, 8);
      t.R = rnd(1, 7);
      t.S = rnd(1, 7);
      t.dh = rnd(1, 3) == 3 ? rnd(2, 3) : 1;
      t.dw = rnd(1, 3) == 3 ? rnd(2, 3) : 1;
      t.sh = rnd(1, 3);
      t.sw = rnd(1, 3);
      t.ph = rnd(0, t.R / 2 + 1);
      t.pw = rnd(0, t.S / 2 + 1);
      t.H = rnd(t.dh * (t.R - 1) + 1, big ? 120 : 40);
      t.W = rnd(t.dw * (t.S - 1) + 1, big ? 120 : 40);
      const int g = rnd(1, 4) == 4 ? rnd(2, 4) : 1;
      t.C = g * (big ? rnd(16, 256) : rnd(1, 48));
      t.K = g * (big ? rnd(16, 384) : rnd(1, 64));
      t.dt = rnd(0, 1);
      t.P = out_dim(t.H, t.ph, t.dh * (t.R - 1) + 1, t.sh);
      t.Q = out_dim(t.W, t.pw, t.dw * (t.S - 1) + 1, t.sw);
      if (t.P < 1 || t.Q < 1 || validate(t) != CONV2D_OK) continue;
      Desc d;
      if (group_desc(t, g, d) != CONV2D_OK) continue;
      ++drawn;
      char nm[96];
      std::snprintf(nm, sizeof nm, "rand%d[%d,%d,%dx%d,%d,%dx%d,p%d%d,s%d%d,d%d%d,g%d,%s]", drawn, t.N, t.C, t.H, t.W,
                    t.K, t.R, t.S, t.ph, t.pw, t.sh, t.sw, t.dh, t.dw, g, t.dt ? "bf16" : "f32");
      void* px = (void*)0x100000;
      void* pw = (void*)0x200000;
      void* py = (void*)0x300000;
      void* ws = (void*)0x400000;
      for (int op = 0; op < 2; ++op) {
        TapSet set;
        const int rc = op == 0 ? build_tap_set(CONV2D_OP_FWD, d, px, pw, py, ws, di, set)
                               : build_tap_set(CONV2D_OP_BWD_DATA, d, py, pw, px, ws, di, set);
        if (rc != CONV2D_OK) {
          fail(nm, op == 0 ? "fwd" : "bwd_data", "no plan");
          continue;
        }
        for (const TapBuild& b : set.pass) {
          check_tap(nm, op == 0 ? "fwd" : "bwd_data", b, di);
          ++plans;
        }
        check_tap_semantics(nm, op == 0 ? "fwd" : "bwd_data", d, set, op == 0);
      }
      WgradBuild bw;
      const int rcw = build_bwd_filter(d, px, py, pw, ws, di, bw);
      const bool phases = phase_need(d, di) != 0;
      if (rcw == CONV2D_OK) {
        check_wgrad(nm, d, bw, di);
        ++plans;
      } else if (rcw != CONV2D_ERR_UNSUPPORTED) {
        fail(nm, "bwd_filter", "planner error");
      } else if (!phases) {
        ++refused;  // the documented refusal: no stage layout fits shared memory
      }
      check_phases(nm, d, di, plans);
    }
  }
  // Layer-scale strided or dilated filter gradients whose slot ring does not fit are refused
  // today (a smaller m-tile group and dilated stride phases would plan them); pin the count so
  // that a change shows here.
  if (refused > 21) fail("random sweep", "bwd_filter", "more refusals than expected");
  std::printf("checked %d plans, %d backward-filter refusals, %d violations\n", plans, refused, g_fail);
  return g_fail > 100 ? 100 : g_fail;
}

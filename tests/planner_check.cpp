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

#include <cmath>
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
  if (p.a_tma) {
    // staged rows as tensor copies of the packed source: equal boxes of at most 128 rows
    // (256 8-byte elements) that tile the rows; one stage's bytes within the barrier's
    // transaction count; copy coordinates (2 per position) within 32 bits
    if (p.rows != p.a_nbox * p.a_box || p.a_box % 8 || p.a_box < 8 || p.a_box > 128)
      fail(nm, op, "tensor-copy boxes do not tile the staged rows");
    // one copy per stage: box (2, rows, NCH, planes of the stage), every dimension at most 256,
    // exactly the stage's A bytes
    const long long planes = p.plane_per_phase ? 1 : p.npl;
    if (p.a_one != (!p.plane_per_phase && p.npl > 1 && p.rows <= 256 ? 1 : 0)) fail(nm, op, "one-copy staging choice");
    if (p.a_one && (planes > 256 || (long long)p.a_stage_bytes % (16ll * p.rows * planes) != 0 ||
                    (long long)p.a_stage_bytes / (16ll * p.rows * planes) > 256))
      fail(nm, op, "one-copy box beyond the copy limits or the stage");
    if ((long long)p.a_stage_bytes + p.b_stage_bytes >= (1 << 20)) fail(nm, op, "stage bytes over the barrier limit");
    if (2 * (p.Mtot + p.rows) >= (1ll << 31)) fail(nm, op, "copy coordinates beyond 32 bits");
    const NhwcPackPlan& q = b.px;
    bool same = q.EX == p.EL && q.WL == p.WL && q.npl == p.npl && q.step_h == p.pl_step_h && q.step_w == p.pl_step_w &&
                q.N == p.N && q.C == p.Cs && q.H == p.Hs && q.W == p.Ws && q.src_nstride == p.src_nstride;
    for (int pl = 0; pl < p.npl; ++pl) same = same && q.off_h[pl] == p.pl_off_h[pl] && q.off_w[pl] == p.pl_off_w[pl];
    if (!same) fail(nm, op, "source pack geometry differs from the tap plan's");
    if (b.src_pack_bytes != (size_t)q.npl * q.nchunk * (size_t)p.Mtot * 16) fail(nm, op, "source pack size");
  }
}

// The channel-chunk pack, run on the host exactly as the kernel walks it (units, staged rows
// and channel runs, output groups), against the definition of the packed planes:
//   dst[pl][cc][n][e][f][j] = src[n][CHUNK*cc + j][e*step_h + off_h[pl]][f*step_w + off_w[pl]]
// (zero outside the source).  Every group must be written once with that value; the source
// holds each element's own index, so a wrong row, column, channel or image shows.  Small
// tensors only (the emulation touches every element).
template <class E>
void check_pack_as_kernel(const char* nm, const char* op, const NhwcPackPlan& q) {
  constexpr int CHUNK = 16 / (int)sizeof(E);
  const long long HW = (long long)q.H * q.W;
  const long long src_elems = (long long)(q.N - 1) * q.src_nstride + (long long)q.C * HW;
  const long long groups = (long long)q.npl * q.nchunk * q.N * q.EX * q.WL;
  if (src_elems > (1ll << 22) || groups > (1ll << 22)) return;
  if (q.units != (unsigned)((long long)q.N * q.ngroups * q.n_etiles) || q.te < 1 ||
      (long long)q.te * q.n_etiles < q.EX || (long long)q.te * (q.n_etiles - 1) >= q.EX || q.cg < 1 ||
      (long long)q.cg * q.ngroups < q.nchunk || (long long)q.cg * (q.ngroups - 1) >= q.nchunk)
    fail(nm, op, "pack units do not tile the padded rows and chunks");
  std::vector<E> src((size_t)src_elems);
  for (size_t i = 0; i < src.size(); ++i) src[i] = (E)(i * 2654435761u + 1u);
  std::vector<E> dst((size_t)groups * CHUNK, (E)0);
  std::vector<int> wrote((size_t)groups, 0);
  std::vector<E> sm((size_t)q.cg * CHUNK * q.ch_pitch);
  for (unsigned v = 0; v < q.units; ++v) {
    const int r = (int)(v / (unsigned)q.n_etiles), et = (int)(v % (unsigned)q.n_etiles);
    const int n = r / q.ngroups, cc0 = (r % q.ngroups) * q.cg, ncc = std::min(q.cg, q.nchunk - cc0);
    const int e0 = et * q.te, ne = std::min(q.te, q.EX - e0);
    const int h_lo = e0 * q.step_h + q.off_h_min, h_hi = (e0 + ne - 1) * q.step_h + q.off_h_min + q.h_span;
    const int hl = std::max(h_lo, 0), hh = std::min(h_hi, q.H - 1), nr = hh - hl + 1;
    const int nchs = std::min(ncc * CHUNK, q.C - CHUNK * cc0);
    // the kernel's transposed staging applies when every channel row starts on a 16-byte
    // boundary (a 16-byte aligned tensor here) and W is a multiple of CHUNK
    const long long row0 = (long long)n * q.src_nstride + (long long)(CHUNK * cc0) * HW + (long long)hl * q.W;
    const bool tr = q.W % CHUNK == 0 && (row0 * (long long)sizeof(E)) % 16 == 0 && (HW * (long long)sizeof(E)) % 16 == 0;
    auto slot = [&](long long pos) { return pos ^ ((pos / CHUNK) & (CHUNK - 1)); };
    if (nr > 0) {
      if ((long long)nr * q.W > q.ch_pitch) {
        fail(nm, op, "pack unit stages more rows than its channel pitch holds");
        return;
      }
      if (tr) {  // region of chunk ccl: ch_pitch position slots of CHUNK channels
        for (int ccl = 0; ccl < ncc; ++ccl)
          for (long long k = 0; k < (long long)nr * q.W; ++k) {
            const long long sl = slot(k);
            if (sl < 0 || sl >= q.ch_pitch) {
              fail(nm, op, "a transposed staging slot leaves its chunk's region");
              return;
            }
            for (int e = 0; e < CHUNK; ++e) {
              const int c = ccl * CHUNK + e;
              sm[((size_t)ccl * q.ch_pitch + (size_t)sl) * CHUNK + e] =
                  c < nchs ? src[(size_t)(row0 + (long long)c * HW + k)] : (E)0;
            }
          }
      } else {
        for (int c = 0; c < nchs; ++c)
          for (long long k = 0; k < (long long)nr * q.W; ++k)
            sm[(size_t)c * q.ch_pitch + k] = src[(size_t)(row0 + (long long)c * HW + k)];
      }
    }
    for (int ccl = 0; ccl < ncc; ++ccl)
      for (int pl = 0; pl < q.npl; ++pl)
        for (int i = 0; i < ne * q.WL; ++i) {
          const int de = i / q.WL, f = i % q.WL;
          const int h = (e0 + de) * q.step_h + q.off_h[pl], w = f * q.step_w + q.off_w[pl];
          const int nch = std::min(CHUNK, nchs - ccl * CHUNK);
          const long long g = (((long long)pl * q.nchunk + cc0 + ccl) * q.N + n) * q.EX * q.WL + (long long)e0 * q.WL + i;
          ++wrote[(size_t)g];
          const bool in = nr > 0 && h >= hl && h <= hh && w >= 0 && w < q.W;
          for (int c = 0; c < CHUNK; ++c) {
            E val = (E)0;
            if (in && tr)
              val = sm[((size_t)ccl * q.ch_pitch + (size_t)slot((long long)(h - hl) * q.W + w)) * CHUNK + c];
            else if (in && c < nch)
              val = sm[(size_t)(ccl * CHUNK + c) * q.ch_pitch + (size_t)(h - hl) * q.W + w];
            dst[(size_t)g * CHUNK + c] = val;
          }
        }
  }
  for (int pl = 0; pl < q.npl; ++pl)
    for (int cc = 0; cc < q.nchunk; ++cc)
      for (int n = 0; n < q.N; ++n)
        for (int e = 0; e < q.EX; ++e)
          for (int f = 0; f < q.WL; ++f) {
            const long long g = ((((long long)pl * q.nchunk + cc) * q.N + n) * q.EX + e) * q.WL + f;
            if (wrote[(size_t)g] != 1) {
              fail(nm, op, "a packed group is not written exactly once");
              return;
            }
            const int h = e * q.step_h + q.off_h[pl], w = f * q.step_w + q.off_w[pl];
            for (int j = 0; j < CHUNK; ++j) {
              const int c = CHUNK * cc + j;
              const E want = (c < q.C && h >= 0 && h < q.H && w >= 0 && w < q.W)
                                 ? src[(size_t)(n * q.src_nstride + (long long)c * HW + (long long)h * q.W + w)]
                                 : (E)0;
              if (dst[(size_t)g * CHUNK + j] != want) {
                fail(nm, op, "a packed element differs from the plane definition");
                return;
              }
            }
          }
}

// bf16 backward-filter on channel-chunked planes: the shared-memory carve of the kernel fits the
// request and the device limit; both packs, run as the kernel walks them, match the plane
// definition; and the plan's tap groups, offsets and output taps, applied to the packed planes
// in fp64, give the filter gradient of the definition (small problems: the emulation sums every
// product).
void check_wgrad_mn(const char* nm, const Desc& d, const DevInfo& di) {
  const char* op = "bwd_filter(mn)";
  MnBuild b;
  alignas(256) static char ws[64];
  const int rc = build_wgrad_mn(d, ws, ws, ws, ws, di, b);
  if (rc == CONV2D_ERR_UNSUPPORTED || rc == CONV2D_ERR_TOO_LARGE) return;
  if (rc != CONV2D_OK) {
    fail(nm, op, "planner error");
    return;
  }
  const WgradMnPlan& p = b.p;
  // carve: 1 KB alignment slack, the stages, 8 epilogue staging tiles of 32 x 80 floats, barriers
  const size_t carve = 1023 + (size_t)p.stages * (p.a_stage_bytes + p.b_stage_bytes) + 8 * 32 * 80 + 8 * (2 * p.stages + 3) + 8;
  if (carve > wgrad_mn_smem_bytes(p)) fail(nm, op, "shared-memory carve beyond the request");
  if (wgrad_mn_smem_bytes(p) > di.smem_optin) fail(nm, op, "shared memory over budget");
  check_pack_as_kernel<uint16_t>(nm, op, b.px);
  check_pack_as_kernel<uint16_t>(nm, op, b.pd);
  const long long M = p.Mtot;
  const long long macs = (long long)d.K * d.C * d.R * d.S * M;
  if (macs > 40000000ll || (long long)d.N * d.C * d.H * d.W > 2000000ll) return;
  std::vector<double> x((size_t)d.N * d.C * d.H * d.W), dy((size_t)d.N * d.K * d.P * d.Q);
  unsigned long long st = 12345;
  auto u = [&]() {  // uniform in [-1, 1), splitmix64
    st += 0x9E3779B97F4A7C15ull;
    unsigned long long z = st;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    return (double)(z >> 11) / (double)(1ull << 52) - 1.0;
  };
  for (double& v : x) v = u();
  for (double& v : dy) v = u();
  auto plane = [&](const NhwcPackPlan& q, const std::vector<double>& src, int pl, int c, long long L) {
    if (L >= M || c >= q.C) return 0.0;
    const long long n = L / ((long long)q.EX * q.WL), rem = L % ((long long)q.EX * q.WL);
    const int h = (int)(rem / q.WL) * q.step_h + q.off_h[pl], w = (int)(rem % q.WL) * q.step_w + q.off_w[pl];
    if (h < 0 || h >= q.H || w < 0 || w >= q.W) return 0.0;
    return src[(((size_t)n * q.C + c) * q.H + h) * q.W + w];
  };
  std::vector<double> dw((size_t)d.K * d.C * d.R * d.S, NAN);
  std::vector<int> seen((size_t)d.R * d.S, 0);
  for (int gi = 0; gi < p.ngroups; ++gi)
    for (int j = 0; j < p.grp_ntaps[gi]; ++j) {
      const int t = p.grp_tap0[gi] + j;
      const int off = p.grp_off0[gi] + p.tap_delta[t];
      if (p.tap_delta[t] + p.KB > p.KBX) fail(nm, op, "tap offset beyond the staged box");
      if (p.tap_out[t] < 0 || p.tap_out[t] >= d.R * d.S) {
        fail(nm, op, "output tap outside the filter");
        return;
      }
      ++seen[(size_t)p.tap_out[t]];
      for (int k = 0; k < d.K; ++k)
        for (int c = 0; c < d.C; ++c) {
          double acc = 0;
          for (long long L = 0; L < M; ++L)
            acc += plane(b.px, x, p.grp_plane[gi], c, L + off) * plane(b.pd, dy, 0, k, L);
          dw[((size_t)k * d.C + c) * d.R * d.S + p.tap_out[t]] = acc;
        }
    }
  for (size_t i = 0; i < seen.size(); ++i)
    if (seen[i] != 1) {
      fail(nm, op, "a filter tap is not produced exactly once");
      return;
    }
  for (int k = 0; k < d.K; ++k)
    for (int c = 0; c < d.C; ++c)
      for (int r = 0; r < d.R; ++r)
        for (int s2 = 0; s2 < d.S; ++s2) {
          double ref = 0;
          for (int n = 0; n < d.N; ++n)
            for (int pp = 0; pp < d.P; ++pp)
              for (int q = 0; q < d.Q; ++q) {
                const int h = pp * d.sh - d.ph + r * d.dh, w = q * d.sw - d.pw + s2 * d.dw;
                if (h < 0 || h >= d.H || w < 0 || w >= d.W) continue;
                ref += x[(((size_t)n * d.C + c) * d.H + h) * d.W + w] * dy[(((size_t)n * d.K + k) * d.P + pp) * d.Q + q];
              }
          const double got = dw[(((size_t)k * d.C + c) * d.R + r) * d.S + s2];
          if (!(std::fabs(got - ref) <= 1e-9 * (1.0 + std::fabs(ref)))) {
            fail(nm, op, "the planned GEMM on the packed planes differs from the definition");
            return;
          }
        }
}

// The workspace of a tap set: the repacked filters of the passes, then (single pass) the packed
// source, 256-byte aligned and inside the set's size.
void check_tap_set(const char* nm, const char* op, const TapSet& set, const void* ws, int dt) {
  if (set.pass.size() != 1 || !set.pass[0].p.a_tma) return;
  const TapBuild& b = set.pass[0];
  const size_t off = static_cast<const uint8_t*>(b.px.dst) - static_cast<const uint8_t*>(ws);
  if (off % 256 || off < b.pack_bytes || off + b.src_pack_bytes != set.pack_bytes)
    fail(nm, op, "packed source misplaced in the workspace");
  if (dt == 1) check_pack_as_kernel<uint16_t>(nm, op, b.px);
  else check_pack_as_kernel<uint32_t>(nm, op, b.px);
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
            if (p.plane_per_phase) {
              // the phase reads the one plane at linear e*WL + f + tap offset + its shift, which may
              // leave the image: there it must land on a zero row or column of the grid (past the
              // source's rows / columns) of a neighbouring image, or before the first / past the
              // last image (zero fill); inside, on the pixel the definition names
              if (fwd || pl != 0) {
                fail(nm, op, "phase shifts outside backward-data with one plane");
                bad = true;
                break;
              }
              const int nh = oh + d.ph - r * d.dh, nw = ow + d.pw - s * d.dw;
              const bool inside = ((nh % d.sh) + d.sh) % d.sh == 0 && ((nw % d.sw) + d.sw) % d.sw == 0;
              if (!inside) {
                fail(nm, op, "a tap sits in a phase whose outputs it does not reach");
                bad = true;
                break;
              }
              const long long dh = floor_div(nh, d.sh), dwc = floor_div(nw, d.sw);
              const bool def_zero = dh < 0 || dh >= p.Hs || dwc < 0 || dwc >= p.Ws;
              const long long img = (long long)p.EL * p.WL;
              for (int n = 0; n < std::min(p.N, 2); ++n) {  // the first image and one after it
                const long long Lr = n * img + (long long)e * p.WL + f + p.tap_off[t] + p.ph_shift[ph];
                bool got_zero = Lr < 0 || Lr >= p.Mtot;
                long long gn = 0, ge = 0, gf = 0;
                if (!got_zero) {
                  gn = Lr / img;
                  ge = (Lr % img) / p.WL;
                  gf = Lr % p.WL;
                  got_zero = ge >= p.Hs || gf >= p.Ws;
                }
                if (got_zero != def_zero || (!got_zero && (gn != n || ge != dh || gf != dwc))) {
                  fail(nm, op, "a shifted phase reads the wrong dy pixel");
                  bad = true;
                  break;
                }
              }
              if (bad) break;
              continue;
            }
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

// The few-channel backward-data kernel (dgrad_c2i_kernel), run on the host exactly as it walks
// its tiles: for the 8 anchor rows x 32 staged columns of a tile, T summed over the row shifts d
// with the kernel's filter operand (tap r with r*dh = d*sh + phi_h, zero outside dy), the column
// fold with the kernel's shift codes (a lane below the shift reads its own value, as the shuffle
// does) and the owned pixels it writes.  Checked against the definition
//   dx[n][c][h][w] = sum over k, r, s with h = p*sh - ph + r*dh, w = q*sw - pw + s*dw of
//                    dy[n][k][p][q] * w[k][c][r][s]   (filter rotated in convolution mode)
// in fp64: every pixel written exactly once, with that value.  Budgets as the launch sees them.
void check_c2i(const char* nm, const Desc& d, const DevInfo& di, int flip, int& plans) {
  C2iPlan p;
  if (build_c2i(d, nullptr, nullptr, nullptr, di, p) != CONV2D_OK) return;
  ++plans;
  if (c2i_smem_bytes(p) > di.smem_optin) fail(nm, "c2i", "shared memory over budget");
  {
    C2iPlan q = p;  // the launch with tensor copies of dy
    q.nraw = q.nraw_tma;
    if (c2i_smem_bytes(q) > di.smem_optin) fail(nm, "c2i", "shared memory over budget (box slots)");
    if (p.nraw_tma != 0 && (d.Q % 4 || (d.P * d.Q) % 4 || p.nraw_tma < 2 || p.nraw_tma > 4))
      fail(nm, "c2i", "box slots");
  }
  if (p.nast < 2 || p.nast > 4) fail(nm, "c2i", "operand slots");
  if (p.Nr % 16 || p.Nr > 128 || p.Nr < d.C * d.sh * 8) fail(nm, "c2i", "MMA N");
  if (p.tmem_cols > 512 || p.tmem_cols < 4 * p.Nr) fail(nm, "c2i", "TMEM columns");
  if (p.TWq < 1 || p.dlt_w > 7 || d.S > 8 || d.sw > 8 || d.sh > 8 || p.EH != 8 + p.dlt_h || p.EH * 32 * 16 >= (1 << 18))
    fail(nm, "c2i", "tile geometry");
  const double work = (double)p.tiles * 256.0 * d.C * d.sh * 8 * (p.dlt_h + 1) * d.K;
  if (work > 3e8) return;  // the emulation below is for small problems
  const int g = d.g;
  const long long dyn = (long long)g * d.K * d.P * d.Q, dxn = (long long)g * d.C * d.H * d.W;
  if (p.dy_nstride != dyn || p.dx_nstride != dxn) fail(nm, "c2i", "image strides");
  std::vector<double> dy((size_t)d.N * dyn), w((size_t)d.K * d.C * d.R * d.S);
  unsigned long long st = 12345;
  auto rnd = [&]() {
    st = st * 6364136223846793005ull + 1442695040888963407ull;
    return (double)((st >> 11) & 0xFFFFF) / 1048576.0 - 0.5;
  };
  for (auto& v : dy) v = rnd();
  for (auto& v : w) v = rnd();
  auto W_ = [&](int k, int c, int r, int s) {
    const int rr = flip ? d.R - 1 - r : r, ss = flip ? d.S - 1 - s : s;
    return w[(((size_t)k * d.C + c) * d.R + rr) * d.S + ss];
  };
  // group 0 of the batch: dy channels 0..K-1, dx channels 0..C-1
  std::vector<double> ref((size_t)d.N * d.C * d.H * d.W, 0.0);
  for (int n = 0; n < d.N; ++n)
    for (int c = 0; c < d.C; ++c)
      for (int h = 0; h < d.H; ++h)
        for (int x = 0; x < d.W; ++x) {
          double acc = 0;
          for (int r = 0; r < d.R; ++r) {
            const int a = h + d.ph - r * d.dh;
            if (a < 0 || a % d.sh) continue;
            const int pp = a / d.sh;
            if (pp >= d.P) continue;
            for (int s = 0; s < d.S; ++s) {
              const int b = x + d.pw - s * d.dw;
              if (b < 0 || b % d.sw) continue;
              const int q = b / d.sw;
              if (q >= d.Q) continue;
              for (int k = 0; k < d.K; ++k) acc += dy[(size_t)n * dyn + ((size_t)k * d.P + pp) * d.Q + q] * W_(k, c, r, s);
            }
          }
          ref[(((size_t)n * d.C + c) * d.H + h) * d.W + x] = acc;
        }
  std::vector<double> out(ref.size(), 0.0);
  std::vector<int> hits(ref.size(), 0);
  unsigned ctab[8];
  for (int phi = 0; phi < 8; ++phi) {
    unsigned code = 0;
    for (int s = 0; s < d.S; ++s) {
      const int dd = s * d.dw - phi;
      if (phi < d.sw && dd >= 0 && dd % d.sw == 0) code |= (8u | (unsigned)(dd / d.sw)) << (4 * s);
    }
    ctab[phi] = code;
  }
  const int ngrp = d.C * d.sh;
  auto dyv = [&](int n, int k, int pp, int q) {
    return (pp < 0 || pp >= d.P || q < 0 || q >= d.Q) ? 0.0 : dy[(size_t)n * dyn + ((size_t)k * d.P + pp) * d.Q + q];
  };
  // filter operand of shift dd, group gi = c*sh + phi_h, tap s (zero where the kernel's is)
  auto Wd = [&](int dd, int k, int gi, int s) {
    const int c = gi / d.sh, phh = gi % d.sh;
    const int rd = dd * d.sh + phh, r = rd / d.dh;
    if (s >= d.S || rd % d.dh || r >= d.R) return 0.0;
    return W_(k, c, r, s);
  };
  std::vector<double> T(32 * 8);
  for (long long t = 0; t < p.tiles; ++t) {
    const long long per = (long long)p.ntp * p.ntq;
    const int n = (int)(t / per), rem = (int)(t % per);
    const int p_lo = p.p_start + (rem / p.ntq) * 8;
    const int q_lo = p.q_start + (rem % p.ntq) * p.TWq - p.dlt_w;
    for (int j = 0; j < 8; ++j)
      for (int gi = 0; gi < ngrp; ++gi) {
        for (int lane = 0; lane < 32; ++lane)
          for (int s = 0; s < 8; ++s) {
            double acc = 0;
            for (int dd = 0; dd <= p.dlt_h; ++dd)
              for (int k = 0; k < d.K; ++k) acc += dyv(n, k, p_lo + j - dd, q_lo + lane) * Wd(dd, k, gi, s);
            T[lane * 8 + s] = acc;
          }
        const int c = gi / d.sh, phh = gi % d.sh;
        const int h = (p_lo + j) * d.sh - d.ph + phh;
        for (int lane = p.dlt_w; lane < 32; ++lane)
          for (int phi = 0; phi < d.sw; ++phi) {
            double acc = 0;
            for (int s = 0; s < 8; ++s) {
              const unsigned code = (ctab[phi] >> (4 * s)) & 15u;
              if (!(code & 8u)) continue;
              const int src = lane >= (int)(code & 7u) ? lane - (int)(code & 7u) : lane;
              acc += T[src * 8 + s];
            }
            const int x = (q_lo + lane) * d.sw - d.pw + phi;
            if (h < 0 || h >= d.H || x < 0 || x >= d.W) continue;
            const size_t o = (((size_t)n * d.C + c) * d.H + h) * d.W + x;
            out[o] = acc;
            ++hits[o];
          }
      }
  }
  int bad_hits = 0, bad_val = 0;
  for (size_t i = 0; i < ref.size(); ++i) {
    if (hits[i] != 1) ++bad_hits;
    else if (std::fabs(out[i] - ref[i]) > 1e-9 * (1.0 + std::fabs(ref[i]))) ++bad_val;
  }
  if (bad_hits) {
    std::printf("  %s c2i: %d pixels not written exactly once\n", nm, bad_hits);
    fail(nm, "c2i", "pixel coverage");
  }
  if (bad_val) {
    std::printf("  %s c2i: %d pixels differ from the definition\n", nm, bad_val);
    fail(nm, "c2i", "folded sums differ from the definition");
  }
}

int main() {
  using namespace cg3;
  // The last field gives the tap passes expected for forward and backward-data.  The tap GEMM
  // stages the filter slices of every tap of a phase for each k-block: in tap-pair mode one
  // 16-byte chunk of source channels per tap (two taps share one MMA), otherwise two or more.
  // A 16x16 stride-1 filter over N = 64 columns is 256 taps x 64 x 16 bytes = 256 KB a stage
  // even in pair mode, so two stages do not fit in shared memory and the taps are split over
  // passes; smaller N or fewer taps fit one pass.  The source channels are C forward and K
  // backward-data; N follows the destination channels (K forward, C backward-data).
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
      {"r15", 1, 4, 40, 40, 8, 15, 15, 7, 7, 1, 1, 0, 1, 1, 1, {1, 1}},
      {"r15_k4", 1, 8, 40, 40, 4, 15, 15, 7, 7, 1, 1, 0, 1, 1, 1, {1, 1}},
      {"r16_c16", 1, 16, 40, 40, 16, 16, 16, 7, 7, 1, 1, 0, 1, 1, 1, {1, 1}},
      {"r16_c32", 1, 32, 40, 40, 32, 16, 16, 7, 7, 1, 1, 0, 1, 1, 1, {2, 2}},
      {"r13_c64", 1, 64, 30, 30, 64, 13, 13, 6, 6, 1, 1, 0, 1, 1, 1, {2, 2}},
      {"r15_bf16_k96", 1, 40, 40, 40, 96, 15, 15, 7, 7, 1, 1, 1, 1, 1, 1, {4, 2}},
      {"r16_s2_bf16", 2, 24, 40, 40, 20, 16, 16, 7, 7, 2, 2, 1, 1, 1, 1, {2, 1}},
      {"r1_s256", 1, 16, 4, 300, 16, 1, 256, 0, 3, 1, 1, 0, 1, 1, 1, {1, 1}},
      {"r1_s256_c64", 1, 64, 4, 300, 64, 1, 256, 0, 3, 1, 1, 0, 1, 1, 1, {3, 3}},
      {"r17", 1, 4, 40, 40, 8, 17, 17, 8, 8, 1, 1, 0, 1, 1, 1, {2, 2}},
      {"r17_bf16", 1, 8, 36, 36, 16, 17, 17, 8, 8, 1, 1, 1, 1, 1, 1, {2, 2}},
      {"s5_patch", 2, 3, 20, 20, 8, 5, 5, 0, 0, 5, 5, 0, 1, 1, 1, {1, 1}},
      {"s6x5", 1, 6, 27, 26, 5, 3, 4, 1, 2, 6, 5, 0, 1, 1, 1, {1, 1}},
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
      // few input channels: backward-data runs the scatter-form kernel where it plans
      {"c2i_stem", 1, 3, 37, 45, 16, 7, 7, 3, 3, 2, 2, 0, 1, 1, 1, {1, 1}},
      {"c2i_s1", 2, 1, 19, 70, 40, 3, 3, 1, 1, 1, 1, 0, 1, 1, 1, {1, 1}},
      {"c2i_dil", 1, 2, 23, 29, 8, 3, 3, 2, 2, 1, 1, 0, 2, 2, 1, {1, 1}},
      {"c2i_s32", 1, 4, 25, 22, 12, 5, 4, 1, 2, 3, 2, 0, 1, 1, 1, {1, 1}},
      {"c2i_k33", 1, 3, 12, 12, 33, 3, 3, 1, 1, 1, 1, 0, 1, 1, 1, {1, 1}},
      {"c2i_r1s8", 1, 4, 9, 40, 20, 1, 8, 0, 3, 1, 1, 0, 1, 1, 1, {1, 1}},
      {"c2i_s4", 1, 2, 18, 37, 7, 4, 4, 0, 1, 4, 4, 0, 1, 1, 1, {1, 1}},
      {"c2i_grp", 2, 6, 11, 13, 10, 3, 3, 1, 1, 2, 1, 0, 1, 1, 2, {1, 1}},
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
      const int rc = op == 0 ? build_tap_set(CONV2D_OP_FWD, d, px, pw, py, ws, di, set, true)
                             : build_tap_set(CONV2D_OP_BWD_DATA, d, py, pw, px, ws, di, set, true);
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
      check_tap_set(s.nm, opn, set, ws, d.dt);
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
    const int rcf = build_bwd_filter(d, px, py, pw, ws, di, bw);
    // backward-filter refuses more than kMaxTaps filter taps (the documented limit)
    if (rcf != CONV2D_OK && !(rcf == CONV2D_ERR_UNSUPPORTED && d.R * d.S > kMaxTaps))
      fail(s.nm, "bwd_filter", "no plan");
    if (rcf == CONV2D_OK && d.R * d.S > kMaxTaps) fail(s.nm, "bwd_filter", "planned past the tap tables");
    check_phases(s.nm, d, di, plans);
    check_c2i(s.nm, d, di, 0, plans);
    check_c2i(s.nm, d, di, 1, plans);
    Desc d16 = d;  // the channel-chunked path plans bf16 only
    d16.dt = 1;
    check_wgrad_mn(s.nm, d16, di);
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
        const int rc = op == 0 ? build_tap_set(CONV2D_OP_FWD, d, px, pw, py, ws, di, set, true)
                               : build_tap_set(CONV2D_OP_BWD_DATA, d, py, pw, px, ws, di, set, true);
        if (rc != CONV2D_OK) {
          fail(nm, op == 0 ? "fwd" : "bwd_data", "no plan");
          continue;
        }
        for (const TapBuild& b : set.pass) {
          check_tap(nm, op == 0 ? "fwd" : "bwd_data", b, di);
          ++plans;
        }
        check_tap_semantics(nm, op == 0 ? "fwd" : "bwd_data", d, set, op == 0);
        check_tap_set(nm, op == 0 ? "fwd" : "bwd_data", set, ws, d.dt);
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
      if (d.dt == 1) check_wgrad_mn(nm, d, di);
    }
  }
  // Layer-scale strided or dilated filter gradients whose slot ring does not fit are refused
  // today (a smaller m-tile group and dilated stride phases would plan them); pin the count so
  // that a change shows here.
  if (refused > 21) fail("random sweep", "bwd_filter", "more refusals than expected");
  // The GPU parity test's two-half-tile bf16 layer (64 x 16 x 64 x 64, K = 64, 3x3 / 2) plans
  // 256-row tiles over four stride-phase planes whose 312 staged rows take one copy per plane and
  // box; the deconvolution forward stages its four planes with one copy.
  {
    auto fwd_plan = [&](int N, int C, int H, int W, int K, int R, int S, int pd, int sd, TapSet& set) {
      Desc d{};
      d.N = N; d.C = C; d.H = H; d.W = W; d.K = K; d.R = R; d.S = S;
      d.ph = pd; d.pw = pd; d.sh = sd; d.sw = sd; d.dt = 1;
      d.P = out_dim(d.H, d.ph, d.R, d.sh);
      d.Q = out_dim(d.W, d.pw, d.S, d.sw);
      return build_tap_set(CONV2D_OP_FWD, d, (void*)0x100000, (void*)0x200000, (void*)0x300000, (void*)0x400000,
                           di, set, true);
    };
    TapSet a, b;
    if (fwd_plan(64, 16, 64, 64, 64, 3, 3, 1, 2, a) != CONV2D_OK || a.pass.size() != 1 || a.pass[0].p.MH != 2 ||
        a.pass[0].p.npl != 4 || a.pass[0].p.a_one != 0 || !a.pass[0].p.a_tma)
      fail("two-half", "fwd", "expected 256-row tiles staged by one copy per plane and box");
    if (fwd_plan(32, 256, 32, 32, 512, 4, 4, 1, 2, b) != CONV2D_OK || b.pass.size() != 1 || b.pass[0].p.a_one != 1)
      fail("deconv", "fwd", "expected one copy per stage");
  }
  std::printf("checked %d plans, %d backward-filter refusals, %d violations\n", plans, refused, g_fail);
  return g_fail > 100 ? 100 : g_fail;
}

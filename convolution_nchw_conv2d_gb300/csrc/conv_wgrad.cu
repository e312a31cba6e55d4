// conv_wgrad.cu -- backward-filter convolution on sm_103a tensor cores.
//
//   dw[k,c,r,s] = sum_{n,p,q} X(n, c, p*sh - ph + r, q*sw - pw + s) * dy[n,k,p,q]
// (the filter gradient of the cuDNN backward-filter call in Apache SystemDS
// LibMatrixCuDNNConvolutionAlgorithm.java; deconvolution's backward-weights in Apache
// MXNet mkldnn_deconvolution.cc is the same product with the weight's roles swapped).
//
// One GEMM per tile (see WgradPlan in conv_plan.h): 128 rows (c, tap) x NK output
// channels k, reduction over a range of the forward linear position space L.
//   producers  stage dy[k, L] per pipeline stage (K-major: positions contiguous, as in
//              NCHW) and append the stage's new x positions to a ring of x rows (one row
//              per plane and channel), so every x position is read from memory once per tile.
//   builders   write the im2col rows A[(c, tap), L] = X_plane(tap)[c, L + tap_off] into
//              TMEM, 32 columns per buffer (tcgen05.st); the 32 lanes of a warp read 32
//              ring rows whose starts fall in distinct shared-memory banks.
//   MMA warp   issues tcgen05.mma with A from TMEM and B = dy from shared memory
//              (kind::tf32 / kind::f16 with bf16), 4 per buffer, accumulating in TMEM.
//   epilogue   stores each tile's fp32 sums as a split partial; a second kernel adds the
//              partials in a fixed order (deterministic) and writes dw in KCRS.
#include "conv_plan.h"
#include "conv_stage.cuh"
#include "sm103_ptx.cuh"

namespace cg3 {

__device__ int g_wgrad_err;

namespace {
// CTA roles (672 threads): warps 0-7 two producer groups taking pipeline stages in turn,
// warps 8-15 two builder sets (set h builds the A buffers with index mod 2 == h), warps
// 16-19 epilogue, warp 20 TMEM allocation + MMA issue.
constexpr int kThreads = 672;
constexpr int kProdThreads = 128;
constexpr int kBuildWarp0 = 8;
constexpr int kEpiWarp0 = 16;
constexpr int kMmaWarp = 20;
constexpr int kNabuf = 4;               // TMEM A buffers of 32 columns
constexpr int kAcol = 32 * kNabuf;      // first accumulator column

__device__ __forceinline__ uint32_t bar_at(uint32_t base, int i) { return base + 8u * (uint32_t)i; }

struct WTile {
  int mt, nt, sp;
};
__device__ __forceinline__ WTile decode_wtile(const WgradPlan& p, long long t) {
  WTile w;
  w.mt = (int)(t % p.n_mtiles);
  long long r = t / p.n_mtiles;
  w.nt = (int)(r % p.n_ntiles);
  w.sp = (int)(r / p.n_ntiles);
  return w;
}

// (channel, tap) of lane `lane` of row unit `unit`; false for a padding row.
__device__ __forceinline__ bool unit_row(const WgradPlan& p, int unit, int lane, int& c, int& tap) {
  c = 0;
  tap = 0;
  if (unit >= p.nunits) return false;
  const int cg = unit / p.upc;
  const int tu = unit - cg * p.upc;
  if (p.TPU == 1) {
    c = cg * p.Cg + lane;
    tap = tu;
    return c < p.C;
  }
  const int tl = lane / p.Cg;
  c = lane - tl * p.Cg;
  tap = tu * p.TPU + tl;
  return tl < p.TPU && tap < p.RS;
}

// First channel of the ring rows of m-tile mt.
__device__ __forceinline__ int tile_c_lo(const WgradPlan& p, int mt) { return ((4 * mt) / p.upc) * p.Cg; }

// Stages tile-relative x positions [q_begin, q_end) of every plane (the tile starts at
// absolute position L0) into the ring for the tile's channels c_lo .. c_lo + xs - 1, in
// whole slot groups of CHUNK slots (a group may also rewrite neighbouring positions with
// their own values, which is harmless).  Item = (plane, slot group, CHUNK channels):
// loaded as CHUNK 16-byte loads (one per channel, CHUNK consecutive pixels) when the
// group's pixels are one aligned run, else element by element, then transposed in
// registers and stored as CHUNK 16-byte shared stores (one per slot); lanes take
// consecutive channel groups, so 8 lanes store 128 contiguous bytes.
template <int DT>
__device__ __forceinline__ void stage_ring(const WgradPlan& p, uint32_t ring, long long L0, int c_lo, int q_begin,
                                           int q_end, int gtid) {
  constexpr int CHUNK = DT == 0 ? 4 : 8;
  constexpr int ESZ = DT == 0 ? 4 : 2;
  constexpr int U = DT == 0 ? 2 : 1;  // items per batch: all loads of a batch precede its stores
  using E = typename std::conditional<DT == 0, uint32_t, uint16_t>::type;
  const E* xg = static_cast<const E*>(p.x);
  const long long HW = (long long)p.H * p.W;
  const int ncg = p.xs / CHUNK;
  const int gbeg = (q_begin + p.sigma) / CHUNK;
  const int ng = (q_end + p.sigma + CHUNK - 1) / CHUNK - gbeg;
  const int ngr = p.rlen / CHUNK;
  const int total = p.npl * ng * ncg;
  for (int it0 = gtid; it0 < total; it0 += 128 * U) {
    uint4 v[U][CHUNK];  // per item: one uint4 per channel holding CHUNK positions
    uint32_t dst[U];
    bool live[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int it = it0 + 128 * u;
      live[u] = it < total;
#pragma unroll
      for (int i = 0; i < CHUNK; ++i) v[u][i] = make_uint4(0u, 0u, 0u, 0u);
      dst[u] = 0u;
      if (!live[u]) continue;
      const int cgp = it % ncg;
      const int rest = it / ncg;
      const int gi = rest % ng;
      const int pl = rest / ng;
      const int g = gbeg + gi;
      const long long La = L0 + (long long)g * CHUNK - p.sigma;  // absolute position of the first slot
      dst[u] = ring + (uint32_t)((((long long)pl * p.rlen + (long long)(g % ngr) * CHUNK) * p.xs + cgp * CHUNK) * ESZ);
      const int c0 = c_lo + cgp * CHUNK;
      bool done = false;
      if (p.vec_x && La >= 0 && La + CHUNK <= p.Mtot) {
        const uint32_t n = fdiv((uint32_t)La, p.fd_img);
        const uint32_t rem = (uint32_t)La - n * p.fd_img.d;
        const int e = (int)fdiv(rem, p.fd_WL);
        const int f = (int)rem - e * p.WL;
        const int h = e * p.pl_step_h + p.pl_off_h[pl];
        const int w = f + p.pl_off_w[pl];
        if (f + CHUNK <= p.WL && (w & (CHUNK - 1)) == 0) {
          done = true;  // one row, aligned: all valid, all outside, or (not here) mixed
          if (h >= 0 && h < p.H && w >= 0 && w + CHUNK <= p.W) {
            const E* s0 = xg + ((long long)n * p.C + c0) * HW + (long long)h * p.W + w;
#pragma unroll
            for (int i = 0; i < CHUNK; ++i)
              if (c0 + i < p.C) v[u][i] = __ldg(reinterpret_cast<const uint4*>(s0 + i * HW));
          } else if (!(w + CHUNK <= 0 || w >= p.W || h < 0 || h >= p.H)) {
            done = false;  // partly inside: element by element
          }
        }
      }
      if (!done) {
#pragma unroll
        for (int j = 0; j < CHUNK; ++j) {
          const long long L = La + j;
          if (L < 0 || L >= p.Mtot) continue;
          const uint32_t n = fdiv((uint32_t)L, p.fd_img);
          const uint32_t rem = (uint32_t)L - n * p.fd_img.d;
          const int e = (int)fdiv(rem, p.fd_WL);
          const int f = (int)rem - e * p.WL;
          const int h = e * p.pl_step_h + p.pl_off_h[pl];
          const int w = f * p.pl_step_w + p.pl_off_w[pl];
          if (h < 0 || h >= p.H || w < 0 || w >= p.W) continue;
          const E* s0 = xg + ((long long)n * p.C + c0) * HW + (long long)h * p.W + w;
#pragma unroll
          for (int i = 0; i < CHUNK; ++i) {
            if (c0 + i >= p.C) break;
            const uint32_t x = (uint32_t)__ldg(s0 + i * HW);
            uint32_t* wv = reinterpret_cast<uint32_t*>(&v[u][i]);
            if constexpr (DT == 0) wv[j] = x;
            else wv[j >> 1] |= x << (16 * (j & 1));
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!live[u]) continue;
#pragma unroll
      for (int j = 0; j < CHUNK; ++j) {
        const uint32_t d = dst[u] + (uint32_t)(j * p.xs * ESZ);
        if constexpr (DT == 0) {
          st_shared_v4(d, comp(v[u][0], j), comp(v[u][1], j), comp(v[u][2], j), comp(v[u][3], j));
        } else {
          const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
          const int k = j >> 1;
          st_shared_v4(d, __byte_perm(comp(v[u][0], k), comp(v[u][1], k), sel),
                       __byte_perm(comp(v[u][2], k), comp(v[u][3], k), sel),
                       __byte_perm(comp(v[u][4], k), comp(v[u][5], k), sel),
                       __byte_perm(comp(v[u][6], k), comp(v[u][7], k), sel));
        }
      }
    }
  }
}

// Position range [lbeg, lend) of split sp.
__device__ __forceinline__ void split_range(const WgradPlan& p, int sp, long long& lbeg, long long& lend) {
  lbeg = (long long)sp * p.split_len;
  lend = lbeg + p.split_len;
  if (lend > p.Mtot) lend = p.Mtot;
}
}  // namespace

template <int DT>
__global__ void __launch_bounds__(kThreads, 1) wgrad_kernel(const __grid_constant__ WgradPlan p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  constexpr int ESZ = DT == 0 ? 4 : 2;
  constexpr int CHUNK = 16 / ESZ;       // elements per 16-byte chunk
  constexpr int PPC = DT == 0 ? 1 : 2;  // positions per TMEM column (and per ring slot)
  constexpr int BUFP = 32 * PPC;        // positions per A buffer
  constexpr int KIND = DT;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int S = p.stages;
  const int KB = p.KB;
  const int nbuf = KB / BUFP;  // A buffers per stage
  const int rlen = p.rlen;

  uint8_t* ptr = smem_raw;
  const uint32_t a0 = smem_u32(ptr);  // dy tiles
  ptr += (size_t)S * p.a_stage_bytes;
  const uint32_t ring = smem_u32(ptr);  // x ring, [plane][slot][xs channels]
  ptr += ((size_t)p.npl * p.rlen * p.xs * ESZ + 15) & ~size_t(15);
  int* tabs = reinterpret_cast<int*>(ptr);  // dy position table per producer group
  ptr += (size_t)2 * KB * sizeof(int);
  ptr = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ptr) + 15) & ~uintptr_t(15));
  const uint32_t full = smem_u32(ptr);
  const uint32_t empty = full + 8u * S;
  const uint32_t afull = empty + 8u * S;
  const uint32_t aempty = afull + 8u * kNabuf;
  const uint32_t accf = aempty + 8u * kNabuf;
  const uint32_t acce = accf + 16u;
  const uint32_t xfree = acce + 16u;
  const uint32_t drain = xfree + 8u;
  ptr += 8 * (2 * S + 2 * kNabuf + 6);
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(ptr);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ptr + 4);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_at(full, s), kProdThreads);
      mbar_init(bar_at(empty, s), 1 + 8);  // MMA commit + 8 builder warps
    }
    for (int b = 0; b < kNabuf; ++b) {
      mbar_init(bar_at(afull, b), 4);  // the 4 warps of the building set
      mbar_init(bar_at(aempty, b), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_at(accf, a), 1);
      mbar_init(bar_at(acce, a), 4);
    }
    mbar_init(xfree, 8);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32((const void*)tmem_holder), (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const long long PQ = (long long)p.P * p.Q;

  if (warp < kBuildWarp0) {
    // =============================================================== producers
    const int grp = warp >> 2;
    const int gtid = tid & (kProdThreads - 1);
    int* dytab = tabs + grp * KB;
    long long counter = 0;
    int ti = 0;  // tiles of this CTA so far
    bool ok = true;
    for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++ti) {
      const WTile wt = decode_wtile(p, t);
      long long lbeg, lend;
      split_range(p, wt.sp, lbeg, lend);
      const int kbase = wt.nt * p.NK;
      const int c_lo = tile_c_lo(p, wt.mt);
      int s_local = 0;
      for (long long l0 = lbeg; l0 < lend; l0 += KB, ++counter, ++s_local) {
        // Stage ownership is a pure function of the counter, so all threads of a group
        // pass the same named barriers even after an abort (which only skips work).
        if ((int)(counter & 1) != grp) continue;
        const int stage = (int)(counter % S);
        const uint32_t ephase = (uint32_t)((counter / S) & 1);
        named_bar_sync(1 + grp, kProdThreads);
        for (int i = gtid; i < KB; i += kProdThreads) {
          const long long L = l0 + i;
          int off = -1;
          if (L < lend) {
            const uint32_t n = fdiv((uint32_t)L, p.fd_img);
            const uint32_t rem = (uint32_t)L - n * p.fd_img.d;
            const int e = (int)fdiv(rem, p.fd_WL);
            const int f = (int)rem - e * p.WL;
            if (e < p.P && f < p.Q) off = (int)((long long)n * p.K * PQ + (long long)e * p.Q + f);
          }
          dytab[i] = off;
        }
        named_bar_sync(1 + grp, kProdThreads);
        if (!ok) continue;
        if (!mbar_wait(bar_at(empty, stage), ephase ^ 1u, abort_flag, &g_wgrad_err)) {
          ok = false;
          continue;
        }
        // The first stages of a tile overwrite ring slots the previous tile's builders
        // may still be reading.
        if (s_local < S && ti > 0 && !mbar_wait(xfree, (uint32_t)((ti - 1) & 1), abort_flag, &g_wgrad_err)) {
          ok = false;
          continue;
        }
        const uint32_t a_st = a0 + (uint32_t)stage * p.a_stage_bytes;
        // dy: [chunk][k row][CHUNK positions]
        stage_position_rows<DT>(p.dy, PQ, dytab, KB / CHUNK, p.NK, p.K - kbase, a_st, kbase, p.vec_dy != 0, gtid);
        // x: this stage's new positions (stage 0 also loads the halo).
        if (s_local == 0)
          stage_ring<DT>(p, ring, lbeg, c_lo, 0, KB + p.max_off, gtid);
        else
          stage_ring<DT>(p, ring, lbeg, c_lo, s_local * KB + p.max_off, (s_local + 1) * KB + p.max_off, gtid);
        cp_async_commit();  // wait_group only covers committed groups
        cp_async_wait<0>();
        fence_proxy_async();
        mbar_arrive(bar_at(full, stage));
      }
    }
    cp_async_commit();
    cp_async_wait<0>();
  } else if (warp < kEpiWarp0) {
    // =============================================================== builders
    const int set = (warp - kBuildWarp0) >> 2;  // builds A buffers with index mod 2 == set
    const int q = warp & 3;                      // TMEM lane quarter
    long long counter = 0, kglob = 0;
    bool ok = true;
    for (long long t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
      const WTile wt = decode_wtile(p, t);
      long long lbeg, lend;
      split_range(p, wt.sp, lbeg, lend);
      int c, tap;
      const bool rv = unit_row(p, wt.mt * 4 + q, lane, c, tap);
      const int c_lo = tile_c_lo(p, wt.mt);
      // byte offset of this lane's (plane, channel) in ring slot 0; slot offset of its tap
      const uint32_t rowb = rv ? (uint32_t)(((long long)p.tap_plane[tap] * p.rlen * p.xs + (c - c_lo)) * ESZ) : 0u;
      const uint32_t sstr = (uint32_t)(p.xs * ESZ);  // bytes per slot
      const int toff = (rv ? p.tap_off[tap] : 0) + p.sigma;
      int sb = 0;  // tile-relative position of the stage's first position, mod rlen
      for (long long l0 = lbeg; l0 < lend && ok; l0 += KB, ++counter) {
        const int stage = (int)(counter % S);
        const uint32_t fphase = (uint32_t)((counter / S) & 1);
        if (!mbar_wait(bar_at(full, stage), fphase, abort_flag, &g_wgrad_err)) {
          ok = false;
          break;
        }
        for (int b = 0; b < nbuf; ++b, ++kglob) {
          if ((int)(kglob & 1) != set) continue;
          const int abuf = (int)(kglob % kNabuf);
          const uint32_t use = (uint32_t)((kglob / kNabuf) & 1);
          if (!mbar_wait(bar_at(aempty, abuf), use ^ 1u, abort_flag, &g_wgrad_err)) {
            ok = false;
            break;
          }
          uint32_t v[32];
          int slot = sb + b * BUFP + toff;
          if (slot >= rlen) slot -= rlen;
          if (rv) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if constexpr (DT == 0) {
                asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v[j]) : "r"(ring + rowb + (uint32_t)slot * sstr));
                slot += 1;
                if (slot >= rlen) slot -= rlen;
              } else {
                uint16_t lo, hi;
                asm volatile("ld.shared.u16 %0, [%1];" : "=h"(lo) : "r"(ring + rowb + (uint32_t)slot * sstr));
                slot += 1;
                if (slot >= rlen) slot -= rlen;
                asm volatile("ld.shared.u16 %0, [%1];" : "=h"(hi) : "r"(ring + rowb + (uint32_t)slot * sstr));
                slot += 1;
                if (slot >= rlen) slot -= rlen;
                v[j] = (uint32_t)lo | ((uint32_t)hi << 16);
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0u;
          }
          tc_fence_after();
          tmem_st32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(abuf * 32), v);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_at(afull, abuf));
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_at(empty, stage));  // done reading this stage's x
        sb += KB;
        if (sb >= rlen) sb -= rlen;
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(xfree);  // the ring may be refilled for the next tile
    }
  } else if (warp < kMmaWarp) {
    // =============================================================== epilogue
    const int q = warp & 3;
    int acc = 0;
    uint32_t aphase = 0;
    for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
      const WTile wt = decode_wtile(p, t);
      if (!mbar_wait(bar_at(accf, acc), aphase, abort_flag, &g_wgrad_err)) break;
      tc_fence_after();
      int c, tap;
      const bool rv = unit_row(p, wt.mt * 4 + q, lane, c, tap);
      const int k0 = wt.nt * p.NK;
      float* dst = p.partial + (((long long)wt.sp * p.RS + tap) * p.C + c) * (long long)p.K + k0;
      const uint32_t tcol = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(kAcol + acc * p.NK);
      const bool vec = (p.K & 3) == 0;
      for (int c0 = 0; c0 < p.NK; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(tcol + (uint32_t)c0, r);
        tmem_ld_wait();
        if (rv) {
          const int kk = k0 + c0;
          if (vec && kk + 16 <= p.K) {
#pragma unroll
            for (int j = 0; j < 16; j += 4)
              *reinterpret_cast<uint4*>(dst + c0 + j) = make_uint4(r[j], r[j + 1], r[j + 2], r[j + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (kk + j < p.K) dst[c0 + j] = __uint_as_float(r[j]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_at(acce, acc));
      if (++acc == p.accb) {
        acc = 0;
        aphase ^= 1u;
      }
    }
  } else {
    // =============================================================== MMA issuer
    // The whole warp runs the loop; one elected lane issues and commits.
    const bool leader = elect_one();
    const uint32_t id = idesc(KIND, 128, p.NK, 0, 0);
    const uint32_t b_hi = (uint32_t)(sdesc(0u, 0u, 128u) >> 32);
    const uint32_t nk16 = (uint32_t)p.NK;  // one chunk of the dy tile, in descriptor units
    long long counter = 0, kglob = 0;
    int acc = 0;
    uint32_t aphase = 0;
    bool ok = true;
    bool issued_any = false;
    for (long long t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
      long long lbeg, lend;
      split_range(p, decode_wtile(p, t).sp, lbeg, lend);
      if (!mbar_wait(bar_at(acce, acc), aphase ^ 1u, abort_flag, &g_wgrad_err)) break;
      tc_fence_after();
      const uint32_t dcol = tmem + (uint32_t)(kAcol + acc * p.NK);
      bool first = true;
      for (long long l0 = lbeg; l0 < lend && ok; l0 += KB, ++counter) {
        const int stage = (int)(counter % S);
        const uint32_t fphase = (uint32_t)((counter / S) & 1);
        if (!mbar_wait(bar_at(full, stage), fphase, abort_flag, &g_wgrad_err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // B = dy tile, K-major [chunk][k row][16 B]; buffer b, MMA i uses chunks 8b+2i, 8b+2i+1.
        const uint32_t blo0 = (uint32_t)sdesc(a0 + (uint32_t)stage * p.a_stage_bytes, (uint32_t)p.NK * 16u, 0u);
        for (int b = 0; b < nbuf; ++b, ++kglob) {
          const int abuf = (int)(kglob % kNabuf);
          const uint32_t use = (uint32_t)((kglob / kNabuf) & 1);
          if (!mbar_wait(bar_at(afull, abuf), use, abort_flag, &g_wgrad_err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (leader) {
            const uint32_t blo = blo0 + (uint32_t)(8 * b) * nk16;
            const uint32_t acol = tmem + (uint32_t)(abuf * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              mma_ts_lh<KIND>(dcol, acol + (uint32_t)(8 * i), blo + (uint32_t)(2 * i) * nk16, b_hi, id,
                              (first && i == 0) ? 0u : 1u);
            tc_commit(bar_at(aempty, abuf));
          }
          __syncwarp();
          issued_any = true;
          first = false;
        }
        if (!ok) break;
        if (leader) tc_commit(bar_at(empty, stage));
      }
      if (!ok) break;
      if (leader) tc_commit(bar_at(accf, acc));
      if (++acc == p.accb) {
        acc = 0;
        aphase ^= 1u;
      }
    }
    if (!ok && issued_any && leader) {
      tc_commit(drain);
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
  }
}

// Sum the split partials in split order and write dw (KCRS).  One thread per
// (tap, c, k) with k fastest, so partial reads are coalesced.
template <int DT>
__global__ void wgrad_reduce_kernel(const __grid_constant__ ReducePlan rp) {
  const int RS = rp.R * rp.S;
  const long long total = (long long)RS * rp.C * rp.K;
  const long long split_stride = (long long)RS * rp.c_pad * rp.k_pad;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int k = (int)(i % rp.K);
    long long r = i / rp.K;
    const int c = (int)(r % rp.C);
    const int tap = (int)(r / rp.C);
    const float* src = rp.partial + ((long long)tap * rp.c_pad + c) * rp.k_pad + k;
    float acc = 0.f;
    for (int s = 0; s < rp.nsplit; ++s) acc += src[s * split_stride];
    const long long o = ((long long)k * rp.C + c) * RS + tap;
    if constexpr (DT == 0)
      static_cast<float*>(rp.dw)[o] = acc;
    else
      static_cast<__nv_bfloat16*>(rp.dw)[o] = __float2bfloat16_rn(acc);
  }
}

size_t wgrad_smem_bytes(const WgradPlan& p, int dt) {
  size_t b = (size_t)p.stages * p.a_stage_bytes;
  b += ((size_t)p.npl * p.rlen * p.xs * (dt == 0 ? 4 : 2) + 15) & ~size_t(15);
  b += (size_t)2 * p.KB * sizeof(int);
  b = (b + 15) & ~size_t(15);
  b += 8 * (2 * p.stages + 2 * kNabuf + 6) + 16;
  return b + 1024;
}

cudaError_t launch_wgrad(const WgradPlan& p, int dt, int grid, cudaStream_t st) {
  const size_t smem = wgrad_smem_bytes(p, dt);
  cudaError_t e;
  if (dt == 0) {
    e = cudaFuncSetAttribute(wgrad_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    wgrad_kernel<0><<<grid, kThreads, smem, st>>>(p);
  } else {
    e = cudaFuncSetAttribute(wgrad_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    wgrad_kernel<1><<<grid, kThreads, smem, st>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_wgrad_reduce(const ReducePlan& rp, int dt, int num_sms, cudaStream_t st) {
  const long long total = (long long)rp.R * rp.S * rp.C * rp.K;
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (dt == 0)
    wgrad_reduce_kernel<0><<<(int)blocks, 256, 0, st>>>(rp);
  else
    wgrad_reduce_kernel<1><<<(int)blocks, 256, 0, st>>>(rp);
  return cudaGetLastError();
}

int wgrad_take_error() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_wgrad_err, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) cudaMemcpyToSymbol(g_wgrad_err, &zero, sizeof(int));
  return v;
}

}  // namespace cg3

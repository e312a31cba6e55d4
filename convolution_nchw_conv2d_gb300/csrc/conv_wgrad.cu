// conv_wgrad.cu -- backward-filter convolution on sm_103a tensor cores.
//
//   dw[k,c,r,s] = sum_{n,p,q} X(n, c, p*sh - ph + r, q*sw - pw + s) * dy[n,k,p,q]
// (the filter gradient of the cuDNN backward-filter call in Apache SystemDS
// LibMatrixCuDNNConvolutionAlgorithm.java; deconvolution's backward-weights in Apache
// MXNet mkldnn_deconvolution.cc is the same product with the weight's roles swapped).
//
// One GEMM per tile (see WgradPlan in conv_plan.h): G m-tiles of 128 rows (c, tap) x NK
// output channels k, reduction over a range of the forward linear position space L.
//   producers  stage dy[k, L] (K-major: positions contiguous, as in NCHW) per pipeline stage,
//              or as a ring of whole linear rows (row-tap sharing), and x either as a ring of
//              whole image rows loaded by tensor copies or as a ring of slots (one row per
//              plane and channel) appended stage by stage, so every x position is read from
//              memory once per tile.
//   builders   write the im2col rows A[(c, tap), L] = X_plane(tap)[c, L + tap_off] into
//              TMEM, 32 columns per buffer (tcgen05.st); the 32 lanes of a warp read 32
//              ring rows whose starts fall in distinct shared-memory banks.
//   MMA warp   issues tcgen05.mma with A from TMEM and B = dy from shared memory
//              (kind::tf32 / kind::f16 with bf16), 4 per buffer -- 4 per filter row sharing
//              the buffer under row-tap sharing -- accumulating in TMEM.
//   epilogue   stores each tile's fp32 sums as a split partial; a second kernel adds the
//              partials in a fixed order (deterministic) and writes dw in KCRS.
#include "conv_plan.h"
#include "conv_stage.cuh"
#include "sm103_ptx.cuh"
#include "launch_util.cuh"

namespace cg3 {

__device__ int g_wgrad_err;

namespace {
// CTA roles: warps 0-3 producers, then kSets builder sets of 4 warps (set h builds the A
// buffers whose running index is h mod kSets), then 4 epilogue warps, then one warp for TMEM
// allocation + MMA issue.
constexpr int kSets = 2;
constexpr int kProdThreads = 128;
constexpr int kBuildWarp0 = 4;
constexpr int kBuildWarps = 4 * kSets;
constexpr int kEpiWarp0 = kBuildWarp0 + kBuildWarps;
constexpr int kMmaWarp = kEpiWarp0 + 4;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr int kNabuf = 4;               // TMEM A buffers of 32 columns
constexpr int kAcol = 32 * kNabuf;      // first accumulator column

__device__ __forceinline__ uint32_t bar_at(uint32_t base, int i) { return base + 8u * (uint32_t)i; }

struct WTile {
  int mg, nt, sp;
  int mt0, gcount;  // first m-tile of the group and the group's m-tiles
};
__device__ __forceinline__ WTile decode_wtile(const WgradPlan& p, long long t) {
  WTile w;
  w.mg = (int)(t % p.n_mgroups);
  long long r = t / p.n_mgroups;
  w.nt = (int)(r % p.n_ntiles);
  w.sp = (int)(r / p.n_ntiles);
  w.mt0 = w.mg * p.G;
  w.gcount = p.n_mtiles - w.mt0 < p.G ? p.n_mtiles - w.mt0 : p.G;
  return w;
}

// (channel, tap) of lane `lane` of row unit `unit`; false for a padding row.
__device__ __forceinline__ bool unit_row(const WgradPlan& p, int unit, int lane, int& c, int& tap) {
  c = 0;
  tap = 0;
  if (unit >= p.nunits) return false;
  const int cg = (int)fdiv((uint32_t)unit, p.fd_upc);
  const int tu = unit - cg * p.upc;
  if (p.TPU == 1) {
    c = cg * p.Cg + lane;
    tap = p.unit_tap[tu];
    return c < p.C;
  }
  const int tl = lane / p.Cg;
  c = lane - tl * p.Cg;
  tap = tu * p.TPU + tl;
  return tl < p.TPU && tap < p.RS;
}

// First channel of the ring rows of a group whose first m-tile is mt0.
__device__ __forceinline__ int tile_c_lo(const WgradPlan& p, int mt0) { return ((4 * mt0) / p.upc) * p.Cg; }

// Stages tile-relative x positions [q_begin, q_end) of every plane (the tile starts at
// absolute position L0) into the ring rows of the tile's channels c_lo .. c_lo + xch - 1,
// in whole slot groups of CHUNK slots (a group may also rewrite neighbouring positions
// with their own values, which is harmless).  Work item = (plane, slot group, block of 8
// rows), spread over all producer threads with the slot group fastest.  A group whose
// pixels are one aligned run (or lie wholly outside the tensor) is one 16-byte cp.async per
// row (zero-filled outside); a mixed group is loaded element by element, a block of rows
// at a time (all loads before the stores).
template <int DT>
__device__ __forceinline__ void stage_ring(const WgradPlan& p, uint32_t ring, long long L0, int c_lo, int q_begin,
                                           int q_end, int gtid) {
  constexpr int CHUNK = DT == 0 ? 4 : 8;
  constexpr int ESZ = DT == 0 ? 4 : 2;
  constexpr int RB = 8;  // rows per item
  using E = typename std::conditional<DT == 0, uint32_t, uint16_t>::type;
  const E* xg = static_cast<const E*>(p.x);
  const long long HW = (long long)p.H * p.W;
  const int gbeg = (q_begin + p.sigma) / CHUNK;
  const int ng = (q_end + p.sigma + CHUNK - 1) / CHUNK - gbeg;
  const int ngr = p.rlen / CHUNK;
  const uint32_t rstride = (uint32_t)(p.xs * ESZ);
  const int nrb = (p.xch + RB - 1) / RB;
  const int total = p.npl * ng * nrb;
  for (int it = gtid; it < total; it += 128) {
    const int gi = it % ng;
    const int rest = it / ng;
    const int rb = rest % nrb;
    const int pl = rest / nrb;
    const int g = gbeg + gi;
    const long long La = L0 + (long long)g * CHUNK - p.sigma;  // absolute position of the first slot
    const uint32_t sdst = ring + (uint32_t)((g % ngr) * CHUNK * ESZ) + (uint32_t)(pl * p.xch) * rstride;
    const int cr0 = rb * RB;
    const int cr1 = cr0 + RB < p.xch ? cr0 + RB : p.xch;
    // classify the group: 1 = one aligned valid run, 2 = all outside, 3 = mixed
    int mode = 3;
    long long soff = 0;
    if (La >= 0 && La + CHUNK <= p.Mtot) {
      const uint32_t n = fdiv((uint32_t)La, p.fd_img);
      const uint32_t rem = (uint32_t)La - n * p.fd_img.d;
      const int e = (int)fdiv(rem, p.fd_WL);
      const int f = (int)rem - e * p.WL;
      if (f + CHUNK <= p.WL) {
        const int h = e * p.pl_step_h + p.pl_off_h[pl];
        const int w = f * p.pl_step_w + p.pl_off_w[pl];
        const int wl = (CHUNK - 1) * p.pl_step_w + w;  // last pixel's column
        if (h < 0 || h >= p.H || wl < 0 || w >= p.W) {
          mode = 2;
        } else if (p.vec_x && (w & (CHUNK - 1)) == 0 && w >= 0 && wl < p.W) {
          mode = 1;
          soff = (long long)n * p.x_nstride + (long long)h * p.W + w;
        }
      }
    }
    if (mode != 3) {
      for (int cr = cr0; cr < cr1; ++cr) {
        const int c = c_lo + cr;
        const bool v = mode == 1 && c < p.C;
        cp_async_16(sdst + (uint32_t)cr * rstride, v ? (const void*)(xg + soff + (long long)c * HW) : p.x, v ? 16 : 0);
      }
      continue;
    }
    // element offsets (channel 0) of the group's positions, -1 = zero
    int offs[CHUNK];
#pragma unroll
    for (int j = 0; j < CHUNK; ++j) {
      offs[j] = -1;
      const long long L = La + j;
      if (L < 0 || L >= p.Mtot) continue;
      const uint32_t nn = fdiv((uint32_t)L, p.fd_img);
      const uint32_t rem = (uint32_t)L - nn * p.fd_img.d;
      const int ee = (int)fdiv(rem, p.fd_WL);
      const int ff = (int)rem - ee * p.WL;
      const int h = ee * p.pl_step_h + p.pl_off_h[pl];
      const int w = ff * p.pl_step_w + p.pl_off_w[pl];
      if (h >= 0 && h < p.H && w >= 0 && w < p.W) offs[j] = (int)((long long)nn * p.x_nstride + (long long)h * p.W + w);
    }
    constexpr int RL = DT == 0 ? 4 : 2;  // rows per load batch
    for (int c0r = cr0; c0r < cr1; c0r += RL) {
      uint32_t wv[RL][4];
#pragma unroll
      for (int r = 0; r < RL; ++r) {
        wv[r][0] = wv[r][1] = wv[r][2] = wv[r][3] = 0u;
        const int c = c_lo + c0r + r;
        if (c0r + r >= cr1 || c >= p.C) continue;
        const E* sc = xg + (long long)c * HW;
#pragma unroll
        for (int j = 0; j < CHUNK; ++j) {
          if (offs[j] < 0) continue;
          const uint32_t x = (uint32_t)__ldg(sc + offs[j]);
          if constexpr (DT == 0) wv[r][j] = x;
          else wv[r][j >> 1] |= x << (16 * (j & 1));
        }
      }
#pragma unroll
      for (int r = 0; r < RL; ++r)
        if (c0r + r < cr1)
          st_shared_v4(sdst + (uint32_t)(c0r + r) * rstride, wv[r][0], wv[r][1], wv[r][2], wv[r][3]);
    }
  }
}

// Stages the dy tile of positions [l0, l0 + KB) (zero at and past lend, and where a
// position has no output) for output channels kbase .. kbase + NK - 1 as the B operand
// [chunk j][k row][16 bytes].  Each warp takes whole chunks (the chunk's class is
// warp-uniform): a chunk of CHUNK valid, contiguous, aligned positions is one 16-byte
// cp.async per row, a chunk with no valid position is zeros, others element by element.
// Rows at and past K - kbase are left untouched (they only reach discarded columns).
template <int DT>
__device__ __forceinline__ void stage_dy(const WgradPlan& p, uint32_t dst0, long long l0, long long lend, int kbase,
                                         int gtid) {
  constexpr int CHUNK = DT == 0 ? 4 : 8;
  using E = typename std::conditional<DT == 0, uint32_t, uint16_t>::type;
  const E* dg = static_cast<const E*>(p.dy);
  const long long PQ = (long long)p.P * p.Q;
  const int lane = gtid & 31, gw = gtid >> 5;
  const int mrows = p.K - kbase < p.NK ? p.K - kbase : p.NK;
  for (int j = gw; j < p.KB / CHUNK; j += 4) {
    const long long La = l0 + (long long)CHUNK * j;
    const uint32_t dbase = dst0 + (uint32_t)(j * p.NK) * 16u;
    int mode = 2;  // 1: 16-byte copies, 2: zeros, 3: element by element
    long long soff = 0;
    if (La < lend) {
      const uint32_t n = fdiv((uint32_t)La, p.fd_img);
      const uint32_t rem = (uint32_t)La - n * p.fd_img.d;
      const int e = (int)fdiv(rem, p.fd_WL);
      const int f = (int)rem - e * p.WL;
      if (p.vec_dy && La + CHUNK <= lend && e < p.P && f + CHUNK <= p.Q) {
        mode = 1;
        soff = (long long)n * p.dy_nstride + (long long)e * p.Q + f;
      } else if (!(p.vec_dy && (e >= p.P || f >= p.Q))) {
        mode = 3;
      }
    }
    if (mode == 1) {
      for (int m = lane; m < mrows; m += 32)
        cp_async_16(dbase + (uint32_t)m * 16u, dg + soff + (long long)(kbase + m) * PQ, 16);
    } else if (mode == 2) {
      for (int m = lane; m < mrows; m += 32) st_shared_v4(dbase + (uint32_t)m * 16u, 0u, 0u, 0u, 0u);
    } else {
      int offs[CHUNK];  // element offsets of the chunk's positions (channel 0), -1 = zero
#pragma unroll
      for (int i = 0; i < CHUNK; ++i) {
        const long long L = La + i;
        offs[i] = -1;
        if (L >= lend) continue;
        const uint32_t n = fdiv((uint32_t)L, p.fd_img);
        const uint32_t rem = (uint32_t)L - n * p.fd_img.d;
        const int e = (int)fdiv(rem, p.fd_WL);
        const int f = (int)rem - e * p.WL;
        if (e < p.P && f < p.Q) offs[i] = (int)((long long)n * p.dy_nstride + (long long)e * p.Q + f);
      }
      // rows in batches of RB: all loads of a batch precede its stores
      constexpr int RB = DT == 0 ? 4 : 2;
      for (int m0 = lane; m0 < mrows; m0 += 32 * RB) {
        uint32_t wv[RB][4];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          wv[r][0] = wv[r][1] = wv[r][2] = wv[r][3] = 0u;
          const int m = m0 + 32 * r;
          if (m >= mrows) continue;
          const E* rowp = dg + (long long)(kbase + m) * PQ;
#pragma unroll
          for (int i = 0; i < CHUNK; ++i) {
            if (offs[i] < 0) continue;
            const uint32_t x = (uint32_t)__ldg(rowp + offs[i]);
            if constexpr (DT == 0) wv[r][i] = x;
            else wv[r][i >> 1] |= x << (16 * (i & 1));
          }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r)
          if (m0 + 32 * r < mrows) st_shared_v4(dbase + (uint32_t)(m0 + 32 * r) * 16u, wv[r][0], wv[r][1], wv[r][2], wv[r][3]);
      }
    }
  }
}

// Position range [lbeg, lend) of split sp.
__device__ __forceinline__ void split_range(const WgradPlan& p, int sp, long long& lbeg, long long& lend) {
  lbeg = (long long)sp * p.split_len;
  lend = lbeg + p.split_len;
  if (lend > p.Mit) lend = p.Mit;
}
}  // namespace

// Bytes of the x ring.
__host__ __device__ inline size_t wgrad_ring_bytes(const WgradPlan& p, int dt) {
  const size_t esz = dt == 0 ? 4 : 2;
  return p.use_tma == 1 ? (size_t)p.NR * p.npl * p.xr * p.WLx * esz : (size_t)p.npl * p.xch * p.xs * esz;
}

// Bytes of the dy row ring (row-tap sharing only).
__host__ __device__ inline size_t wgrad_dyring_bytes(const WgradPlan& p, int dt) {
  const size_t esz = dt == 0 ? 4 : 2;
  return p.TRU > 1 ? (size_t)p.NRd * p.WL * p.NK * esz : 0;
}

// One A buffer's MMAs under row-tap sharing: for each row tap j, the 4 MMAs of the buffer
// (8 * PPC positions each) into accumulator j, with B = dy at the buffer's positions moved
// back by j linear rows, read from the dy row ring ([row slot][chunk][k][16 B]; an MMA's two
// chunks never straddle a row since rows are whole pairs of chunks).  row0 / col0: ring row
// slot and column of the buffer's first position.
template <int KIND, int TRU>
__device__ __forceinline__ void issue_row_taps(const WgradPlan& p, uint32_t dcol, uint32_t acol, uint32_t dyring,
                                               int row0, int col0, uint32_t b_hi, uint32_t id, bool first) {
  constexpr int CHUNK = KIND == 0 ? 4 : 8;
  constexpr int KM = KIND == 0 ? 8 : 16;  // positions per MMA
  const uint32_t cbytes = (uint32_t)p.NK * 16u;         // one chunk of NK rows
  const uint32_t rbytes = (uint32_t)(p.WL / CHUNK) * cbytes;  // one ring row
  const uint32_t lbo = ((cbytes >> 4) & 0x3FFFu) << 16;
  if (col0 + 3 * KM < p.WL) {
    // the buffer's positions lie in one ring row: descriptors advance by one chunk pair per
    // MMA from the row slot of each row tap (computed first, so the MMAs issue back to back)
    uint32_t lo[TRU];
#pragma unroll
    for (int j = 0; j < TRU; ++j) {
      int sl = row0 - j * p.tru_step;
      if (sl < 0) sl += p.NRd;
      lo[j] = (((dyring + (uint32_t)sl * rbytes + (uint32_t)(col0 / CHUNK) * cbytes) & 0x3FFFFu) >> 4) | lbo;
    }
    const uint32_t step = (2u * cbytes) >> 4;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < TRU; ++j)
        mma_ts_lh<KIND>(dcol + (uint32_t)(j * p.NK), acol + (uint32_t)(8 * i), lo[j] + (uint32_t)i * step, b_hi, id,
                        (first && i == 0) ? 0u : 1u);
    return;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int col = col0 + KM * i, row = row0;
    while (col >= p.WL) {  // (rows may be narrower than a buffer)
      col -= p.WL;
      if (++row == p.NRd) row = 0;
    }
    const uint32_t cofs = (uint32_t)(col / CHUNK) * cbytes;
#pragma unroll
    for (int j = 0; j < TRU; ++j) {
      int sl = row - j * p.tru_step;
      if (sl < 0) sl += p.NRd;
      const uint32_t addr = dyring + (uint32_t)sl * rbytes + cofs;
      mma_ts_lh<KIND>(dcol + (uint32_t)(j * p.NK), acol + (uint32_t)(8 * i), ((addr & 0x3FFFFu) >> 4) | lbo, b_hi, id,
                      (first && i == 0) ? 0u : 1u);
    }
  }
}

// tcgen05.st of w[K .. K + 31] to 32 TMEM columns (K fixed, so w stays in registers).
template <int K>
__device__ __forceinline__ void tmem_st32_at(uint32_t taddr, const uint32_t (&w)[36]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(w[K + 0]), "r"(w[K + 1]), "r"(w[K + 2]), "r"(w[K + 3]), "r"(w[K + 4]), "r"(w[K + 5]), "r"(w[K + 6]),
      "r"(w[K + 7]), "r"(w[K + 8]), "r"(w[K + 9]), "r"(w[K + 10]), "r"(w[K + 11]), "r"(w[K + 12]), "r"(w[K + 13]),
      "r"(w[K + 14]), "r"(w[K + 15]), "r"(w[K + 16]), "r"(w[K + 17]), "r"(w[K + 18]), "r"(w[K + 19]),
      "r"(w[K + 20]), "r"(w[K + 21]), "r"(w[K + 22]), "r"(w[K + 23]), "r"(w[K + 24]), "r"(w[K + 25]),
      "r"(w[K + 26]), "r"(w[K + 27]), "r"(w[K + 28]), "r"(w[K + 29]), "r"(w[K + 30]), "r"(w[K + 31])
      : "memory");
}

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
  griddep_launch_dependents();  // the reduce may be scheduled now; it waits for this grid
  const int rlen = p.rlen;

  // 1024-byte aligned base (the size includes the slack): tensor-copy destinations
  uint8_t* ptr = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t a0 = smem_u32(ptr);  // dy tiles per stage, or the dy row ring (TRU > 1)
  ptr += (size_t)S * p.a_stage_bytes + wgrad_dyring_bytes(p, DT);
  const uint32_t ring = smem_u32(ptr);  // x: slot ring [plane][channel][xs], or the row ring (use_tma 1)
  ptr += (wgrad_ring_bytes(p, DT) + 15) & ~size_t(15);
  // per builder warp, m-tile and lane: {ring offset of the lane's row (bit 31: padding row),
  // tap offset} -- set once per tile
  uint2* btab = reinterpret_cast<uint2*>(ptr);
  ptr += (size_t)kBuildWarps * p.G * 32 * sizeof(uint2);
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
      mbar_init(bar_at(empty, s), 1 + kBuildWarps);  // MMA commit + every builder warp
    }
    for (int b = 0; b < kNabuf; ++b) {
      mbar_init(bar_at(afull, b), 4);  // the 4 warps of the building set
      mbar_init(bar_at(aempty, b), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_at(accf, a), 1);
      mbar_init(bar_at(acce, a), 4);
    }
    mbar_init(xfree, kBuildWarps);
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

  if (warp < kBuildWarp0) {
    // =============================================================== producers
    if (p.use_tma) {
      // Copy-engine staging: per stage, one tensor copy per 16-byte chunk of positions
      // (all NK output channels) for dy; for x either tensor copies of whole image rows
      // into the row ring (use_tma 1) or, into the slot ring, one bulk copy per (plane,
      // linear row, channel) for the valid pixel run plus shared stores of zeros for padding
      // slots (use_tma 2).  Every thread adds its own copies' bytes to the stage's full
      // barrier before issuing them and then arrives without waiting, so the producers run
      // ahead by up to S stages.
      const int gtid = tid;
      using E = typename std::conditional<DT == 0, uint32_t, uint16_t>::type;
      const E* xg = static_cast<const E*>(p.x);
      uint32_t last_phase[4] = {0u, 0u, 0u, 0u};  // 1 + parity of the last fill per slot (thread 0)
      long long counter = 0;
      int ti = 0;
      bool ok = true;
      for (long long t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x, ++ti) {
        const WTile wt = decode_wtile(p, t);
        long long lbeg, lend;
        split_range(p, wt.sp, lbeg, lend);
        const int kbase = wt.nt * p.NK;
        const int c_lo = tile_c_lo(p, wt.mt0);
        const int nch_x = p.C - c_lo < p.xch ? p.C - c_lo : p.xch;  // ring rows with real channels
        // Row bookkeeping in 32 bits with multiply-high divisions (positions and rows < 2^31):
        // the producers' issue time is on the pipeline's critical path.
        int next_row = (int)fdiv((uint32_t)(lbeg + p.delta), p.fd_WL);  // first x row not loaded
        int next_dy_row = (int)fdiv((uint32_t)lbeg, p.fd_WL) - (p.TRU - 1) * p.tru_step;  // first dy row not loaded
        int s_local = 0;
        for (long long l0 = lbeg; l0 < lend; l0 += KB, ++counter, ++s_local) {
          const int stage = (int)(counter % S);
          const uint32_t ephase = (uint32_t)((counter / S) & 1);
          if (!mbar_wait(bar_at(empty, stage), ephase ^ 1u, abort_flag, &g_wgrad_err)) {
            ok = false;
            break;
          }
          if (s_local < S && ti > 0 && !mbar_wait(xfree, (uint32_t)((ti - 1) & 1), abort_flag, &g_wgrad_err)) {
            ok = false;
            break;
          }
          // dy row ring: a new tile's rows may map to ring slots of the previous tile's last
          // stages, so every earlier fill must be consumed first (fill c completes phase c / S
          // of its slot's empty barrier; no later phase can have completed yet)
          if (p.TRU > 1 && s_local == 0 && ti > 0) {
            for (long long c = counter - S + 1 > 0 ? counter - S + 1 : 0; c < counter && ok; ++c)
              if (!mbar_wait(bar_at(empty, (int)(c % S)), (uint32_t)((c / S) & 1), abort_flag, &g_wgrad_err))
                ok = false;
            if (!ok) break;
          }
          // the slot's previous contents were read through the generic proxy (builder
          // loads): order those reads before this stage's copy-engine writes
          fence_proxy_async();
          const uint32_t fb = bar_at(full, stage);
          const uint32_t a_st = a0 + (uint32_t)stage * p.a_stage_bytes;
          if (p.TRU > 1) {
            // dy: the linear rows this stage reads that are not loaded yet, from (TRU - 1) * tru_step rows
            // before the stage to its last position; one tensor copy per row (NK channels,
            // [chunk][k][CHUNK]); rows before the first image, past the last one, or past
            // the output height read as zeros.
            const int rdB = (int)fdiv((uint32_t)(l0 + KB - 1), p.fd_WL);
            const int nrows = next_dy_row <= rdB ? rdB - next_dy_row + 1 : 0;
            const uint32_t rbytes = (uint32_t)(p.WL * p.NK * ESZ);
            for (int it = gtid; it < nrows; it += kProdThreads) {
              const int R = next_dy_row + it;
              int n = 0, e = R, slot = R + p.NRd;  // R < 0: a row before the tensor (R > -NRd)
              if (R >= 0) {
                n = (int)fdiv((uint32_t)R, p.fd_EL);
                e = R - n * p.EL;
                slot = R - (int)fdiv((uint32_t)R, p.fd_NRd) * p.NRd;
              }
              mbar_expect_tx(fb, rbytes);
              tma_load_5d(a0 + (uint32_t)slot * rbytes, &p.tm_dyr, 0, kbase, 0, e, n, fb);
            }
            if (nrows > 0) next_dy_row = rdB + 1;
          } else
          // dy: chunk j = positions l0 + CHUNK*j .. +CHUNK-1 (one linear row: WL % CHUNK == 0)
          // chunk j is issued by lane j / 4 of warp j % 4 (the issue work is spread over the
          // four schedulers)
          for (int jb = 0; jb < KB / CHUNK; jb += kProdThreads) {
            const int j = jb + 4 * (gtid & 31) + (gtid >> 5);
            if (j >= KB / CHUNK) continue;
            const long long La = l0 + (long long)CHUNK * j;
            int n = p.N, e = 0, f = 0;  // past the tensor: the copy reads zeros
            if (La < p.Mtot) {
              const uint32_t nn = fdiv((uint32_t)La, p.fd_img);
              const uint32_t rem = (uint32_t)La - nn * p.fd_img.d;
              n = (int)nn;
              e = (int)fdiv(rem, p.fd_WL);
              f = (int)rem - e * p.WL;
            }
            mbar_expect_tx(fb, (uint32_t)(p.NK * 16));
            tma_load_4d(a_st + (uint32_t)(j * p.NK * 16), &p.tm_dy, f, kbase, e, n, fb);
          }
          if (p.use_tma == 1) {
            // x: the linear rows holding this stage's slots that are not loaded yet (one tensor
            // copy per (row, plane, 32 channels)); rows past the tensor read as zeros.
            {
              const int rB = (int)fdiv((uint32_t)(l0 + KB + p.max_off - 1 + p.delta), p.fd_WL);
              if (next_row <= rB) {
                const int nrows = rB - next_row + 1;
                const int ncg = p.xr / 32;
                const int items = nrows * p.npl * ncg;
                for (int it = gtid; it < items; it += kProdThreads) {
                  const int cg = it % ncg;
                  const int rest = it / ncg;
                  const int pl = rest % p.npl;
                  const int R = next_row + rest / p.npl;
                  const int n = (int)fdiv((uint32_t)R, p.fd_EL);
                  const int e = R - n * p.EL;
                  const int h = e * p.pl_step_h + p.pl_off_h[pl];
                  const int rs = R - (int)fdiv((uint32_t)R, p.fd_NR) * p.NR;
                  const uint32_t dst = ring + (uint32_t)(((rs * p.npl + pl) * p.xr + 32 * cg) * p.WLx * ESZ);
                  mbar_expect_tx(fb, (uint32_t)(32 * p.WLx * ESZ));
                  tma_load_4d(dst, &p.tm_x, p.pl_off_w[pl] - p.delta, h, c_lo + 32 * cg, n, fb);
                }
                next_row = rB + 1;
              }
            }
          } else {
            // x: tile-relative positions [q0, q1) (stage 0 also loads the halo); 32-bit
            // position arithmetic (positions < 2^31), divisions by multiply-high
            const int q0 = s_local == 0 ? 0 : s_local * KB + p.max_off;
            const int q1 = (s_local + 1) * KB + p.max_off;
            const uint32_t Lx0 = (uint32_t)(lbeg + q0);
            const uint32_t Lx1 = (uint32_t)(lbeg + q1 < p.Mtot ? lbeg + q1 : p.Mtot);
            const uint32_t lb = (uint32_t)lbeg;
            // slot of tile-relative position q >= -sigma (a copy widened to an aligned start
            // may begin a few positions before the tile: those slots are dead at its start)
            auto slot_of = [&](int q) {
              const uint32_t v = (uint32_t)(q + p.sigma + rlen);
              return (int)(v - fdiv(v, p.fd_rlen) * (uint32_t)rlen);
            };
            if (Lx0 < Lx1) {
              const uint32_t row0 = fdiv(Lx0, p.fd_WL);
              const int nseg = (int)(fdiv(Lx1 - 1u, p.fd_WL) - row0 + 1u);
              const int items = p.npl * nseg * nch_x;
              for (int it = gtid; it < items; it += kProdThreads) {
                const int cr = it % nch_x;
                const int rest = it / nch_x;
                const int sg = rest % nseg;
                const int pl = rest / nseg;
                const uint32_t R = row0 + (uint32_t)sg;  // linear row (image n, row e)
                const uint32_t Rs = R * (uint32_t)p.WL;  // its first position
                const int f0 = (int)((Lx0 > Rs ? Lx0 : Rs) - Rs);
                const int f1 = (int)((Lx1 < Rs + (uint32_t)p.WL ? Lx1 : Rs + (uint32_t)p.WL) - Rs);
                const int n = (int)fdiv(R, p.fd_EL);
                const int e = (int)R - n * p.EL;
                const int h = e * p.pl_step_h + p.pl_off_h[pl];
                const int ow = p.pl_off_w[pl];
                const bool hv = h >= 0 && h < p.H;
                const int rq = (int)(Rs - lb);             // tile-relative position of the row start
                int lo = f0 + ow < 0 ? 0 : f0 + ow;        // valid pixel run [lo, hi)
                int hi = f1 + ow > p.W ? p.W : f1 + ow;
                const uint32_t rowbase = ring + (uint32_t)((pl * p.xch + cr) * p.xs) * ESZ;
                if (hv && lo < hi) {
                  const int wa = lo & ~(CHUNK - 1);
                  const int wb = (hi + CHUNK - 1) & ~(CHUNK - 1);  // <= W (W % CHUNK == 0)
                  const int slot = slot_of(rq + (wa - ow));
                  const E* src = xg + (long long)n * p.x_nstride + ((long long)(c_lo + cr) * p.H + h) * p.W + wa;
                  const int len = wb - wa;
                  const int part = rlen - slot < len ? rlen - slot : len;
                  mbar_expect_tx(fb, (uint32_t)(len * ESZ));
                  bulk_g2s(rowbase + (uint32_t)(slot * ESZ), src, (uint32_t)(part * ESZ), fb);
                  if (part < len) bulk_g2s(rowbase, src + part, (uint32_t)((len - part) * ESZ), fb);
                } else {
                  lo = hi = f1 + ow;  // no valid pixel: every slot of the segment is zero
                }
                // zeros: the segment's positions before and after the valid run
                auto zero_slots = [&](int fa, int fz) {
                  if (fa >= fz) return;
                  int sl = slot_of(rq + fa);
                  for (int ff = fa; ff < fz; ++ff) {
                    if constexpr (DT == 0)
                      asm volatile("st.shared.b32 [%0], %1;" ::"r"(rowbase + (uint32_t)sl * 4u), "r"(0u) : "memory");
                    else
                      asm volatile("st.shared.b16 [%0], %1;" ::"r"(rowbase + (uint32_t)sl * 2u), "h"((uint16_t)0) : "memory");
                    if (++sl == rlen) sl = 0;
                  }
                };
                zero_slots(f0, lo - ow);
                zero_slots(hi - ow, f1);
              }
            }
            // positions past the last image: zeros (they only meet zero dy, but stale
            // shared memory could hold non-finite values)
            if ((long long)lbeg + q1 > p.Mtot) {
              const int za = (int)((Lx0 > (uint32_t)p.Mtot ? (long long)Lx0 : p.Mtot) - lbeg);
              const int nz = q1 - za;
              const int rows = p.npl * p.xch;
              for (int it = gtid; it < nz * rows; it += kProdThreads) {
                const int row = it / nz;
                const int q = za + it - row * nz;
                const uint32_t a = ring + (uint32_t)(row * p.xs + slot_of(q)) * ESZ;
                if constexpr (DT == 0)
                  asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(0u) : "memory");
                else
                  asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"((uint16_t)0) : "memory");
              }
            }
          }
          mbar_arrive(fb);
          if (gtid == 0) last_phase[stage] = 1u + ephase;
        }
      }
      // After an abort, wait (bounded) for copies still in flight into shared memory.
      if (gtid == 0 && *abort_flag) {
        for (int st = 0; st < S; ++st)
          if (last_phase[st]) mbar_wait_drain(bar_at(full, st), last_phase[st] - 1u);
      }
    } else {
    // Stage s's copies are issued, committed as one cp.async group, and its full barrier
    // is arrived on once the next stage's copies are in flight too (wait_group 1), so two
    // stages load at once.  Before any wait that needs the consumers to finish the pending
    // stage (the ring refill at a tile start), the pending stage is completed first.
    const int gtid = tid;
    long long counter = 0;
    int ti = 0;  // tiles of this CTA so far
    int pending = -1;  // stage slot issued but not yet arrived on
    bool ok = true;
    auto complete_pending = [&](bool all) {
      if (pending < 0) return;
      if (all) cp_async_wait<0>();
      else cp_async_wait<1>();
      fence_proxy_async();
      mbar_arrive(bar_at(full, pending));
      pending = -1;
    };
    for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++ti) {
      const WTile wt = decode_wtile(p, t);
      long long lbeg, lend;
      split_range(p, wt.sp, lbeg, lend);
      const int kbase = wt.nt * p.NK;
      const int c_lo = tile_c_lo(p, wt.mt0);
      int s_local = 0;
      for (long long l0 = lbeg; l0 < lend && ok; l0 += KB, ++counter, ++s_local) {
        const int stage = (int)(counter % S);
        const uint32_t ephase = (uint32_t)((counter / S) & 1);
        if (!mbar_wait(bar_at(empty, stage), ephase ^ 1u, abort_flag, &g_wgrad_err)) {
          ok = false;
          break;
        }
        // The first stages of a tile overwrite ring slots the previous tile's builders may
        // still be reading.
        if (s_local < S && ti > 0) {
          complete_pending(true);
          if (!mbar_wait(xfree, (uint32_t)((ti - 1) & 1), abort_flag, &g_wgrad_err)) {
            ok = false;
            break;
          }
        }
        const uint32_t a_st = a0 + (uint32_t)stage * p.a_stage_bytes;
        stage_dy<DT>(p, a_st, l0, lend, kbase, gtid);
        // x: this stage's new positions (stage 0 also loads the halo).
        if (s_local == 0)
          stage_ring<DT>(p, ring, lbeg, c_lo, 0, KB + p.max_off, gtid);
        else
          stage_ring<DT>(p, ring, lbeg, c_lo, s_local * KB + p.max_off, (s_local + 1) * KB + p.max_off, gtid);
        cp_async_commit();
        complete_pending(false);
        pending = stage;
      }
      if (!ok) break;
    }
    complete_pending(true);
    cp_async_wait<0>();
    }
  } else if (warp < kEpiWarp0) {
    // =============================================================== builders
    const int set = (warp - kBuildWarp0) >> 2;  // builds A buffers with running index mod kSets == set
    const int q = warp & 3;                      // TMEM lane quarter
    uint2* mytab = btab + (size_t)(warp - kBuildWarp0) * p.G * 32;
    const uint32_t rslot = (uint32_t)(p.npl * p.xr * p.WLx);  // row ring: elements per row slot
    const int ngr = rlen / CHUNK;
    long long counter = 0, kglob = 0;
    int kset = 0;  // kglob mod kSets
    bool ok = true;
    for (long long t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
      const WTile wt = decode_wtile(p, t);
      long long lbeg, lend;
      split_range(p, wt.sp, lbeg, lend);
      const int c_lo = tile_c_lo(p, wt.mt0);
      // This lane's row of every m-tile of the group: where it lives in the ring and its tap
      // offset (row ring: linear rows << 16 | columns; slot ring: slots).  With one tap per
      // unit the tap, hence the offset, is the same in every lane, padding lanes included.
      for (int g = 0; g < wt.gcount; ++g) {
        int c, tap;
        const bool rv = unit_row(p, (wt.mt0 + g) * 4 + q, lane, c, tap);
        uint32_t off = 0x80000000u, toff = 0u;
        if (p.use_tma == 1) {
          if (rv) off = (uint32_t)((p.tap_plane[tap] * p.xr + (c - c_lo)) * p.WLx);
          if (p.TPU == 1 || rv) toff = (uint32_t)p.tap_rc[tap];
        } else {
          if (rv) off = (uint32_t)((p.tap_plane[tap] * p.xch + (c - c_lo)) * p.xs * ESZ);
          toff = (uint32_t)(((p.TPU == 1 || rv) ? p.tap_off[tap] : 0) + p.sigma);
        }
        mytab[g * 32 + lane] = make_uint2(off, toff);
      }
      __syncwarp();
      int sb = 0;  // slot ring: tile-relative position of the stage's first position, mod rlen
      for (long long l0 = lbeg; l0 < lend && ok; l0 += KB, ++counter) {
        const int stage = (int)(counter % S);
        const uint32_t fphase = (uint32_t)((counter / S) & 1);
        if (!mbar_wait(bar_at(full, stage), fphase, abort_flag, &g_wgrad_err)) {
          ok = false;
          break;
        }
        // row ring: linear row slot and column of the stage's first slot
        int rs0 = 0, c0 = 0;
        if (p.use_tma == 1) {
          const uint32_t sg = (uint32_t)(l0 + p.delta);
          const uint32_t r0 = fdiv(sg, p.fd_WL);
          c0 = (int)(sg - r0 * (uint32_t)p.WL);
          rs0 = (int)(r0 - fdiv(r0, p.fd_NR) * (uint32_t)p.NR);
        }
        int bs_rs = rs0, bs_c = c0;  // row ring position of buffer b's first column
        for (int bg = 0, b = 0, g = 0; bg < nbuf * wt.gcount && ok;
             ++bg, ++kglob, kset = kset + 1 == kSets ? 0 : kset + 1) {
          // b: buffer of positions, g: m-tile within the group (g fastest)
          if (bg > 0 && ++g == wt.gcount) {
            g = 0;
            ++b;
            bs_c += BUFP;
            while (bs_c >= p.WL) {
              bs_c -= p.WL;
              if (++bs_rs == p.NR) bs_rs = 0;
            }
          }
          if (kset != set) continue;
          const int abuf = (int)(kglob & (kNabuf - 1));
          const uint32_t use = (uint32_t)((kglob / kNabuf) & 1);
          if (!mbar_wait(bar_at(aempty, abuf), use ^ 1u, abort_flag, &g_wgrad_err)) {
            ok = false;
            break;
          }
          const uint2 ent = mytab[g * 32 + lane];
          const bool rv = (ent.x & 0x80000000u) == 0u;
          // ring position of this buffer's first column for this lane's tap
          int slot = 0, rs = 0, col = 0;
          if (p.use_tma == 1) {
            col = bs_c + (int)(ent.y & 0xffffu);
            rs = bs_rs + (int)(ent.y >> 16);
            if (col >= p.WL) {
              col -= p.WL;
              ++rs;
            }
            if (rs >= p.NR) rs -= p.NR;
          } else {
            slot = sb + b * BUFP + (int)ent.y;
            while (slot >= rlen) slot -= rlen;
          }
          uint32_t w[36];
          const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(abuf * 32);
          // tcgen05.st is warp-collective: every lane must reach the same instruction, so the
          // read paths below branch on plan values (uniform), never on lane data.
          if (p.TPU == 1) {
            // One tap per unit: the position is the same in all lanes.  9 aligned 16-byte
            // reads cover the 32 columns wherever they start in a group; column j is word
            // k + j (fp32) or halfwords rho + 2j, rho + 2j + 1 (bf16, shifted down when rho is
            // odd).  Groups never straddle ring rows (rlen and WL are chunk multiples).
            const int rho = (p.use_tma == 1 ? col : slot) & (CHUNK - 1);
            const int k = DT == 0 ? rho : rho >> 1;
            if (rv) {
              if (p.use_tma == 1) {
                int cidx = col - rho;
#pragma unroll
                for (int i = 0; i < 9; ++i) {
                  const uint32_t a = ring + ((uint32_t)rs * rslot + ent.x + (uint32_t)cidx) * ESZ;
                  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                               : "=r"(w[4 * i]), "=r"(w[4 * i + 1]), "=r"(w[4 * i + 2]), "=r"(w[4 * i + 3])
                               : "r"(a));
                  cidx += CHUNK;
                  if (cidx == p.WL) {
                    cidx = 0;
                    if (++rs == p.NR) rs = 0;
                  }
                }
              } else {
                int gq = slot / CHUNK;
#pragma unroll
                for (int i = 0; i < 9; ++i) {
                  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                               : "=r"(w[4 * i]), "=r"(w[4 * i + 1]), "=r"(w[4 * i + 2]), "=r"(w[4 * i + 3])
                               : "r"(ring + ent.x + (uint32_t)(gq * 16)));
                  if (++gq == ngr) gq = 0;
                }
              }
              if (DT != 0 && (rho & 1)) {
#pragma unroll
                for (int j = 0; j < 35; ++j) w[j] = __byte_perm(w[j], w[j + 1], 0x5432);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 36; ++j) w[j] = 0u;
            }
            tc_fence_after();
            switch (k) {
              case 0: tmem_st32_at<0>(ta, w); break;
              case 1: tmem_st32_at<1>(ta, w); break;
              case 2: tmem_st32_at<2>(ta, w); break;
              default: tmem_st32_at<3>(ta, w); break;
            }
          } else {
            // Several taps per unit: each lane reads its own positions element by element.
#pragma unroll
            for (int j = 0; j < 36; ++j) w[j] = 0u;
            if (rv) {
#pragma unroll
              for (int j = 0; j < 32 * PPC; ++j) {
                uint32_t a;
                if (p.use_tma == 1) {
                  a = ring + ((uint32_t)rs * rslot + ent.x + (uint32_t)col) * ESZ;
                  if (++col == p.WL) {
                    col = 0;
                    if (++rs == p.NR) rs = 0;
                  }
                } else {
                  a = ring + ent.x + (uint32_t)slot * ESZ;
                  if (++slot == rlen) slot = 0;
                }
                if constexpr (DT == 0) {
                  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w[j]) : "r"(a));
                } else {
                  uint16_t h;
                  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(a));
                  w[j >> 1] |= (uint32_t)h << (16 * (j & 1));
                }
              }
            }
            tc_fence_after();
            tmem_st32_at<0>(ta, w);
          }
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
      const int k0 = wt.nt * p.NK;
      const bool vec = (p.K & 3) == 0;
      for (int gj = 0; gj < wt.gcount * p.TRU; ++gj) {
        // accumulator gj = (m-tile g, row tap j): taps (r0 + j, s) of the unit's base tap
        const int g = gj / p.TRU, j = gj - g * p.TRU;
        int c, tap;
        bool rv = unit_row(p, (wt.mt0 + g) * 4 + q, lane, c, tap);
        if (j > 0) {
          rv = rv && (p.tap_rc[tap] >> 16) + j < p.R;
          tap += j * p.S;
        }
        float* dst = p.partial + (((long long)wt.sp * p.RS + tap) * p.C + c) * (long long)p.K + k0;
        const uint32_t tcol =
            tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(kAcol + ((acc * p.G + g) * p.TRU + j) * p.NK);
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
      const WTile wt = decode_wtile(p, t);
      long long lbeg, lend;
      split_range(p, wt.sp, lbeg, lend);
      if (!mbar_wait(bar_at(acce, acc), aphase ^ 1u, abort_flag, &g_wgrad_err)) break;
      tc_fence_after();
      const uint32_t dcol0 = tmem + (uint32_t)(kAcol + acc * p.G * p.TRU * p.NK);
      bool first_stage = true;
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
        for (int bg = 0, b = 0, g = 0; bg < nbuf * wt.gcount; ++bg, ++kglob) {
          if (bg > 0 && ++g == wt.gcount) {
            g = 0;
            ++b;
          }
          const int abuf = (int)(kglob % kNabuf);
          const uint32_t use = (uint32_t)((kglob / kNabuf) & 1);
          if (!mbar_wait(bar_at(afull, abuf), use, abort_flag, &g_wgrad_err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (leader) {
            const uint32_t acol = tmem + (uint32_t)(abuf * 32);
            const bool first = first_stage && b == 0;
            if (p.TRU == 1) {
              const uint32_t blo = blo0 + (uint32_t)(8 * b) * nk16;
              const uint32_t dcol = dcol0 + (uint32_t)(g * p.NK);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                mma_ts_lh<KIND>(dcol, acol + (uint32_t)(8 * i), blo + (uint32_t)(2 * i) * nk16, b_hi, id,
                                (first && i == 0) ? 0u : 1u);
            } else {
              // ring row slot and column of the buffer's first position
              const uint32_t P0 = (uint32_t)(l0 + (long long)b * BUFP);
              const uint32_t R0 = fdiv(P0, p.fd_WL);
              const int col0 = (int)(P0 - R0 * (uint32_t)p.WL);
              const int row0 = (int)(R0 - fdiv(R0, p.fd_NRd) * (uint32_t)p.NRd);
              const uint32_t dcol = dcol0 + (uint32_t)(g * p.TRU * p.NK);
              switch (p.TRU) {
                case 2: issue_row_taps<KIND, 2>(p, dcol, acol, a0, row0, col0, b_hi, id, first); break;
                case 3: issue_row_taps<KIND, 3>(p, dcol, acol, a0, row0, col0, b_hi, id, first); break;
                default: issue_row_taps<KIND, 4>(p, dcol, acol, a0, row0, col0, b_hi, id, first); break;
              }
            }
            tc_commit(bar_at(aempty, abuf));
          }
          __syncwarp();
          issued_any = true;
        }
        first_stage = false;
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

// Sum the split partials and write dw (KCRS), in a fixed order (deterministic).  A block
// of 8 warps takes 32 * V consecutive outputs (tap, c, k) with k fastest (V = 4 when K is a
// multiple of 4: one 16-byte read per lane, so a warp reads 512 contiguous bytes of a
// split); warp w adds splits w, w + 8, w + 16, ... in order, with the reads of up to 8 of
// its splits issued before their adds, and the 8 warp sums are then added in warp order.
constexpr int kReduceWarps = 8;
template <int DT, int V>
__global__ void __launch_bounds__(32 * kReduceWarps) wgrad_reduce_kernel(const __grid_constant__ ReducePlan rp) {
  __shared__ float part[kReduceWarps][32 * V];
  const int RS = rp.R * rp.S;
  const long long total = (long long)RS * rp.C * rp.K;
  const long long split_stride = (long long)RS * rp.c_pad * rp.k_pad;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  griddep_wait();  // the partials are written by the previous grid
  for (long long o0 = (long long)blockIdx.x * 32 * V; o0 < total; o0 += (long long)gridDim.x * 32 * V) {
    const long long i = o0 + (long long)lane * V;  // first of this lane's V outputs
    float acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = 0.f;
    if (i < total) {
      // partial index of output i: the partial layout [split][tap][c][k] equals the output
      // order (tap, c, k) when c_pad == C and k_pad == K
      const float* src = rp.partial + i;
      int sp = w;
      for (; sp + 7 * kReduceWarps < rp.nsplit; sp += 8 * kReduceWarps) {
        float r[8][V];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float* q = src + (long long)(sp + u * kReduceWarps) * split_stride;
          if constexpr (V == 4) {
            const float4 f = __ldg(reinterpret_cast<const float4*>(q));
            r[u][0] = f.x, r[u][1] = f.y, r[u][2] = f.z, r[u][3] = f.w;
          } else {
            r[u][0] = __ldg(q);
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
          for (int v = 0; v < V; ++v) acc[v] += r[u][v];
      }
      for (; sp < rp.nsplit; sp += kReduceWarps) {
        const float* q = src + (long long)sp * split_stride;
        if constexpr (V == 4) {
          const float4 f = __ldg(reinterpret_cast<const float4*>(q));
          acc[0] += f.x, acc[1] += f.y, acc[2] += f.z, acc[3] += f.w;
        } else {
          acc[0] += __ldg(q);
        }
      }
    }
#pragma unroll
    for (int v = 0; v < V; ++v) part[w][lane * V + v] = acc[v];
    __syncthreads();
    // thread t finalises output o0 + t (t < 32 * V)
    for (int t = threadIdx.x; t < 32 * V; t += 32 * kReduceWarps) {
      const long long io = o0 + t;
      if (io < total) {
        float sum = part[0][t];
#pragma unroll
        for (int j = 1; j < kReduceWarps; ++j) sum += part[j][t];
        const int k = (int)(io % rp.K);
        const long long r = io / rp.K;
        const int c = (int)(r % rp.C);
        const int tap = (int)(r / rp.C);
        int rr = rp.r0 + rp.rstep * (tap / rp.S), ss = rp.s0 + rp.sstep * (tap % rp.S);
        if (rp.flip) {
          rr = rp.R_out - 1 - rr;
          ss = rp.S_out - 1 - ss;
        }
        int cw = c, cn = rp.C;
        if (rp.gk != 0) {  // grouped: keep the diagonal block of k's group
          const int g = k / rp.gk;
          if (c / rp.gc != g) continue;
          cw = c - g * rp.gc;
          cn = rp.gc;
        }
        const long long o = (((long long)k * cn + cw) * rp.R_out + rr) * rp.S_out + ss;
        if constexpr (DT == 0) {
          float* dwp = static_cast<float*>(rp.dw);
          if (rp.beta != 0.f) sum += rp.beta * dwp[o];
          dwp[o] = sum;
        } else {
          __nv_bfloat16* dwp = static_cast<__nv_bfloat16*>(rp.dw);
          if (rp.beta != 0.f) sum += rp.beta * __bfloat162float(dwp[o]);
          dwp[o] = __float2bfloat16_rn(sum);
        }
      }
    }
    __syncthreads();
  }
}

// Per-channel sums (bias gradients) of up to two tensors in one launch (plan `a`, then plan `b`
// when b.t is not NULL).  Block (ch, j) of a plan adds t[n, ch, 0 .. HW) for the images
// n = j*ipb .. j*ipb + ipb - 1: thread i takes the blocks' 16-byte groups i, i + 256, ... in
// order, eight reads in flight (elements instead of groups when HW is not a multiple of a group
// or the tensor is not 16-byte aligned); the 256 thread sums are added by a fixed tree into
// part[ch * nblk + j].  The final pass adds a channel's nblk partials in order, so the sums are
// the same on every run.  (A bf16 value is the high half of the fp32 with the same bits.)
constexpr int kSumThreads = 256;

template <int DT>
__device__ __forceinline__ float sum_group(const uint4& u) {
  const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if constexpr (DT == 0) {
      acc += __uint_as_float(wv[e]);
    } else {
      acc += __uint_as_float(wv[e] << 16);
      acc += __uint_as_float(wv[e] & 0xffff0000u);
    }
  }
  return acc;
}

template <int DT>
__global__ void __launch_bounds__(kSumThreads) chan_sum_partial_kernel(const __grid_constant__ ChanSumPlan a,
                                                                       const __grid_constant__ ChanSumPlan b) {
  __shared__ float red[kSumThreads];
  const long long na = (long long)a.Ch * a.nblk;
  const bool first = blockIdx.x < na;
  const ChanSumPlan& cp = first ? a : b;
  const long long bi = first ? blockIdx.x : blockIdx.x - na;
  const int j = (int)(bi % cp.nblk);
  const int ch = (int)(bi / cp.nblk);
  const int n0 = j * cp.ipb, n1 = min(cp.N, n0 + cp.ipb);
  float acc = 0.f;
  constexpr int VE = DT == 0 ? 4 : 8;  // elements per 16-byte read
  const bool vec = (cp.HW % VE) == 0 && (reinterpret_cast<uintptr_t>(cp.t) & 15) == 0;
  if (vec) {
    // 32-bit group indices within the block (a block reads at most a few hundred KB)
    const uint32_t ng = (uint32_t)(cp.HW / VE);  // groups per image
    const uint32_t tot = ng * (uint32_t)(n1 - n0);
    const uint4* src = reinterpret_cast<const uint4*>(cp.t) + (((long long)n0 * cp.Ch + ch) * cp.HW) / VE;
    const long long istride = (long long)cp.Ch * cp.HW / VE;  // groups from one image to the next
    for (uint32_t g0 = threadIdx.x; g0 < tot; g0 += 8 * kSumThreads) {
      uint4 u[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t g = g0 + (uint32_t)q * kSumThreads;
        u[q] = make_uint4(0u, 0u, 0u, 0u);
        if (g < tot) {
          const uint32_t n = g / ng;
          u[q] = __ldg(src + n * istride + (g - n * ng));
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) acc += sum_group<DT>(u[q]);
    }
  } else {
    const long long tot = cp.HW * (n1 - n0);
    for (long long i = threadIdx.x; i < tot; i += kSumThreads) {
      const long long n = n0 + i / cp.HW, k = i % cp.HW;
      const long long o = (n * cp.Ch + ch) * cp.HW + k;
      if constexpr (DT == 0)
        acc += static_cast<const float*>(cp.t)[o];
      else
        acc += __bfloat162float(static_cast<const __nv_bfloat16*>(cp.t)[o]);
    }
  }
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int h = kSumThreads / 2; h > 0; h >>= 1) {
    if ((int)threadIdx.x < h) red[threadIdx.x] += red[threadIdx.x + h];
    __syncthreads();
  }
  if (threadIdx.x == 0) cp.part[(long long)ch * cp.nblk + j] = red[0];
}

template <int DT>
__global__ void __launch_bounds__(kSumThreads) chan_sum_final_kernel(const __grid_constant__ ChanSumPlan a,
                                                                     const __grid_constant__ ChanSumPlan b) {
  const int i = blockIdx.x * kSumThreads + threadIdx.x;
  const bool first = i < a.Ch;
  const ChanSumPlan& cp = first ? a : b;
  const int ch = first ? i : i - a.Ch;
  if (ch >= cp.Ch || cp.t == nullptr) return;
  float sum = 0.f;
  for (int j = 0; j < cp.nblk; ++j) sum += cp.part[(long long)ch * cp.nblk + j];
  if constexpr (DT == 0) {
    float* o = static_cast<float*>(cp.out);
    if (cp.beta != 0.f) sum += cp.beta * o[ch];
    o[ch] = sum;
  } else {
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(cp.out);
    if (cp.beta != 0.f) sum += cp.beta * __bfloat162float(o[ch]);
    o[ch] = __float2bfloat16_rn(sum);
  }
}

// Sums of a and (b.t not NULL) b; ipb and nblk are set by chan_sum_blocks.
cudaError_t launch_chan_sum(const ChanSumPlan& a, const ChanSumPlan& b, int dt, cudaStream_t st) {
  const long long blocks = (long long)a.Ch * a.nblk + (b.t != nullptr ? (long long)b.Ch * b.nblk : 0ll);
  const long long chs = (long long)a.Ch + (b.t != nullptr ? b.Ch : 0);
  const unsigned fblocks = (unsigned)((chs + kSumThreads - 1) / kSumThreads);
  if (dt == 0) {
    chan_sum_partial_kernel<0><<<(unsigned)blocks, kSumThreads, 0, st>>>(a, b);
    chan_sum_final_kernel<0><<<fblocks, kSumThreads, 0, st>>>(a, b);
  } else {
    chan_sum_partial_kernel<1><<<(unsigned)blocks, kSumThreads, 0, st>>>(a, b);
    chan_sum_final_kernel<1><<<fblocks, kSumThreads, 0, st>>>(a, b);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------- space to depth
// xs[n][a*sw + b][c][i][j] = x[n][c][i*sh + a][j*sw + b], zero outside x.  One (image, plane,
// channel) slab per block row; threads take consecutive j, so stores are contiguous and a
// warp's loads touch sw times its width of one input row.
template <int DT>
__global__ void __launch_bounds__(256) space_to_depth_kernel(const __grid_constant__ S2dPlan sp, int band,
                                                             int nbands) {
  // A unit is one band of `band` rows of every phase plane of one (image, channel): the
  // band's band*sh input rows are one contiguous run, read with coalesced loads into shared
  // memory; each phase plane's rows of the band are then written as one contiguous run.
  extern __shared__ __align__(16) uint8_t s2d_smem[];
  using E = typename std::conditional<DT == 0, uint32_t, uint16_t>::type;
  E* tile = reinterpret_cast<E*>(s2d_smem);
  const E* x = static_cast<const E*>(sp.x);
  E* xs = static_cast<E*>(sp.xs);
  const int npl = sp.sh * sp.sw;
  const long long plane = (long long)sp.Hp * sp.Wp;
  const long long units = (long long)sp.N * sp.C * nbands;
  for (long long u = blockIdx.x; u < units; u += gridDim.x) {
    const int bd = (int)(u % nbands);
    const long long nc = u / nbands;  // n * C + c
    const int c = (int)(nc % sp.C);
    const long long n = nc / sp.C;
    const int i0 = bd * band;
    const int bi = min(band, sp.Hp - i0);
    const int h0 = i0 * sp.sh;
    const int nh = max(0, min(bi * sp.sh, sp.H - h0));
    const E* src = x + nc * (long long)sp.H * sp.W + (long long)h0 * sp.W;
    for (int e = threadIdx.x; e < nh * sp.W; e += blockDim.x) tile[e] = src[e];
    __syncthreads();
    const int per = bi * sp.Wp;
    for (int e = threadIdx.x; e < npl * per; e += blockDim.x) {
      const int pl = e / per;
      const int r = e - pl * per;
      const int ii = r / sp.Wp, j = r - ii * sp.Wp;
      const int a = pl / sp.sw, b = pl - a * sp.sw;
      const int hh = ii * sp.sh + a, w = j * sp.sw + b;
      const E v = (hh < nh && w < sp.W) ? tile[hh * sp.W + w] : E(0);
      xs[((n * npl + pl) * sp.C + c) * plane + (long long)(i0 + ii) * sp.Wp + j] = v;
    }
    __syncthreads();
  }
}

cudaError_t launch_space_to_depth(const S2dPlan& sp, int dt, int num_sms, cudaStream_t st) {
  const int esz = dt == 0 ? 4 : 2;
  const long long row_bytes = (long long)sp.sh * sp.W * esz;  // input bytes per band row
  const int band = (int)std::max(1ll, std::min<long long>(sp.Hp, (16 * 1024) / std::max(1ll, row_bytes)));
  const int nbands = (sp.Hp + band - 1) / band;
  const size_t smem = (size_t)band * row_bytes;
  const long long units = (long long)sp.N * sp.C * nbands;
  const unsigned grid = (unsigned)std::max(1ll, std::min<long long>(units, (long long)num_sms * 16));
  static std::atomic<int> set_bytes[2][kMaxDevices];
  cudaError_t e;
  if (dt == 0) {
    e = ensure_dyn_smem(space_to_depth_kernel<0>, smem, set_bytes[0]);
    if (e != cudaSuccess) return e;
    space_to_depth_kernel<0><<<grid, 256, smem, st>>>(sp, band, nbands);
  } else {
    e = ensure_dyn_smem(space_to_depth_kernel<1>, smem, set_bytes[1]);
    if (e != cudaSuccess) return e;
    space_to_depth_kernel<1><<<grid, 256, smem, st>>>(sp, band, nbands);
  }
  return cudaGetLastError();
}

size_t wgrad_smem_bytes(const WgradPlan& p, int dt) {
  size_t b = (size_t)p.stages * p.a_stage_bytes + wgrad_dyring_bytes(p, dt);
  b += (wgrad_ring_bytes(p, dt) + 15) & ~size_t(15);
  b += (size_t)kBuildWarps * p.G * 32 * sizeof(uint2);
  b = (b + 15) & ~size_t(15);
  b += 8 * (2 * p.stages + 2 * kNabuf + 6) + 16;
  return b + 1024;
}

static std::atomic<int> g_smem_set_0[kMaxDevices], g_smem_set_1[kMaxDevices];

cudaError_t launch_wgrad(const WgradPlan& p, int dt, int grid, cudaStream_t st) {
  const size_t smem = wgrad_smem_bytes(p, dt);
  cudaError_t e;
  if (dt == 0) {
    e = ensure_dyn_smem(wgrad_kernel<0>, smem, g_smem_set_0);
    if (e != cudaSuccess) return e;
    wgrad_kernel<0><<<grid, kThreads, smem, st>>>(p);
  } else {
    e = ensure_dyn_smem(wgrad_kernel<1>, smem, g_smem_set_1);
    if (e != cudaSuccess) return e;
    wgrad_kernel<1><<<grid, kThreads, smem, st>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_wgrad_reduce(const ReducePlan& rp, int dt, int num_sms, cudaStream_t st) {
  const long long total = (long long)rp.R * rp.S * rp.C * rp.K;
  // 16-byte partial reads need every output group of 4 to start on a 16-byte boundary
  const bool v4 = rp.K % 4 == 0 && rp.c_pad == rp.C && rp.k_pad == rp.K &&
                  (reinterpret_cast<uintptr_t>(rp.partial) & 15) == 0;
  const int per_block = 32 * (v4 ? 4 : 1);
  long long blocks = (total + per_block - 1) / per_block;
  const long long cap = (long long)num_sms * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  // programmatic stream serialization: launched while the GEMM runs, waits for it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(32 * kReduceWarps);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (v4)
    e = dt == 0 ? cudaLaunchKernelEx(&cfg, wgrad_reduce_kernel<0, 4>, rp)
                : cudaLaunchKernelEx(&cfg, wgrad_reduce_kernel<1, 4>, rp);
  else
    e = dt == 0 ? cudaLaunchKernelEx(&cfg, wgrad_reduce_kernel<0, 1>, rp)
                : cudaLaunchKernelEx(&cfg, wgrad_reduce_kernel<1, 1>, rp);
  return e != cudaSuccess ? e : cudaGetLastError();
}

int wgrad_take_error() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_wgrad_err, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) cudaMemcpyToSymbol(g_wgrad_err, &zero, sizeof(int));
  return v;
}

}  // namespace cg3

// conv_dgrad_c2i.cu -- backward-data (= deconvolution forward) for problems with few input
// channels C, where the tap GEMM's N dimension (C) would leave the tensor cores mostly idle.
//
// The backward-data sum (page "LibMatrixCuDNNConvolutionAlgorithm.java", the backward-data
// algorithm and its descriptors; page "mkldnn_deconvolution.cc", the deconvolution forward that
// is the same operation): dy element (k, p, q) meets filter tap (c, r, s) once and lands on dx
// pixel (c, p*sh - ph + r*dh, q*sw - pw + s*dw).  Write a dx row as h = p*sh - ph + phi_h
// (p the "anchor" dy row, phi_h < sh its row phase) and a column as w = q*sw - pw + phi_w.
// Filter row r reaches row (p, phi_h) from dy row p - d exactly when r*dh = d*sh + phi_h, and
// filter column s reaches column (q, phi_w) from dy column q - e when s*dw = e*sw + phi_w.  So
//     T[(p, q), (c, phi_h, s)] = sum over d and k of dy[k, p - d, q] * w[k, c, (d*sh + phi_h)/dh, s]
//     dx[c, (p, phi_h), (q, phi_w)] = sum over s of T[(p, q - e(s)), (c, phi_h, s)].
// The first line runs on the tensor cores: for each row shift d one GEMM over k whose A operand
// is the staged dy tile moved back by d whole rows (a start-address offset of the shared-memory
// operand, no copy), all shifts accumulating into one TMEM accumulator (tf32 inputs, fp32 sums;
// filter rows of the shifts that do not exist are zero).  The second line is a fold across the
// lanes of a warp: lane q holds T at dy column q, and a warp shuffle brings the value of column
// q - e to it (ascending s, a fixed order).
//
// Tile: 8 anchor dy rows x 32 dy columns (M = 256, two 128-row MMAs), dy staged from row
// p_lo - dlt_h (dlt_h = the largest row shift).  Columns dlt_w..31 (dlt_w = the largest column
// shift) receive every contribution from inside the tile; tiles step by 32 - dlt_w columns and 8
// rows, so every dx pixel is written once by one tile, straight from registers.
//
// Staging: dy enters shared memory in its own layout, one tensor copy per stage (16 channels x
// EH rows x 36 columns, zero outside the tensor); builder warps read it along positions
// (conflict-free) and write the K-major operand (16 bytes = 4 channels of one position).
// Where dy's rows are not 16-byte aligned (Q or P*Q not a multiple of 4) the builders read dy
// from global memory instead.  Roles: warps 0-3 build; warps 4-5 issue the MMAs (one 128-row
// half each); warps 6-13 fold and store, one TMEM lane quarter and half each; warp 14 issues
// the tensor copies.  Two TMEM accumulators let the MMAs of the next tile run during the
// fold.  Every wait is bounded.
#include <algorithm>
#include <cstdint>

#include <cuda_runtime.h>

#include "conv_plan.h"
#include "conv_stage.cuh"
#include "launch_util.cuh"
#include "sm103_ptx.cuh"

namespace cg3 {

__device__ int g_c2i_err;

namespace {

constexpr int kKS = 16;                    // dy channels per stage (4 chunks of 4)
constexpr int kThreads = 15 * 32;
constexpr int kMmaWarp = 4;                // warps 4 and 5: one 128-row half each
constexpr int kEpiWarp0 = 6;               // warps 6..13: fold and store
constexpr int kCopyWarp = 14;              // warp 14: the dy tensor copies
constexpr int kGB = 6;                     // (c, phi_h) groups per TMEM load batch of the fold

// Each thread of the warp reads 8 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}

struct Tile {
  int n, p_lo, q_lo;  // image; first anchor dy row; dy column of staged lane 0
};

__device__ __forceinline__ Tile tile_of(const C2iPlan& p, long long t) {
  const long long per = (long long)p.ntp * p.ntq;
  Tile c;
  c.n = (int)(t / per);
  const int rem = (int)(t - (long long)c.n * per);
  const int tp = rem / p.ntq, tq = rem - tp * p.ntq;
  c.p_lo = p.p_start + tp * 8;
  c.q_lo = p.q_start + tq * p.TWq - p.dlt_w;
  return c;
}

__device__ __forceinline__ int floor4(int v) { return v >= 0 ? (v & ~3) : -((-v + 3) & ~3); }

// Column fold of one (c, phi_h): out[phi_w] = sum over taps s (ascending) that land on column
// phase phi_w of T at lane - (s*dw - phi_w)/sw.  SW, DW > 0: stride and dilation known at compile
// time (every condition and shift a constant; the padded taps s >= S are summed too, their T
// columns being exactly zero), so the fold has no branches.  SW = 0: any stride and dilation,
// through the per-phase code table (4 bits per tap: bit 3 = lands, bits 0-2 = lane shift).
template <int SW, int DW>
__device__ __forceinline__ void fold_columns(const uint32_t (&z)[8], float (&out)[8], int sw,
                                             const uint32_t (&ctab)[8]) {
  if constexpr (SW > 0) {
#pragma unroll
    for (int phi = 0; phi < SW; ++phi) {
      float acc = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int d = s * DW - phi;
        if (d < 0 || d % SW != 0) continue;
        acc += d == 0 ? __uint_as_float(z[s]) : __shfl_up_sync(0xffffffffu, __uint_as_float(z[s]), (unsigned)(d / SW));
      }
      out[phi] = acc;
    }
  } else {
#pragma unroll
    for (int phi = 0; phi < 8; ++phi) {
      if (phi >= sw) break;
      float acc = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint32_t code = (ctab[phi] >> (4 * s)) & 15u;
        if (code & 8u) acc += __shfl_up_sync(0xffffffffu, __uint_as_float(z[s]), code & 7u);
      }
      out[phi] = acc;
    }
  }
}

}  // namespace

template <int SW, int DW>
__global__ void __launch_bounds__(kThreads, 1) dgrad_c2i_kernel(const __grid_constant__ C2iPlan p) {
  extern __shared__ __align__(16) uint8_t c2i_smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int EH = p.EH;
  const int raw_bytes = 36 * EH * kKS * 4;

  // ---- shared memory: filter operand | staged operands | dy boxes | barriers
  uint8_t* ptr = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(c2i_smem) + 127) & ~uintptr_t(127));
  const uint32_t b0 = smem_u32(ptr);
  ptr += p.b_bytes;
  const uint32_t a0 = smem_u32(ptr);
  ptr += (size_t)p.nast * p.a_bytes;
  const float* raw = reinterpret_cast<const float*>(ptr);
  const uint32_t raw0 = smem_u32(ptr);
  ptr += (size_t)p.nraw * raw_bytes;
  const uint32_t rfull = smem_u32(ptr);    // per dy box slot: the tensor copy landed
  const uint32_t rempty = rfull + 8u * 4;  // per box slot: the four builder warps read it
  const uint32_t afull = rempty + 8u * 4;  // per operand slot: built (four builder warps)
  const uint32_t aempty = afull + 8u * 4;  // per operand slot: both issuing warps' MMAs read it
  const uint32_t tfull = aempty + 8u * 4;  // per accumulator: both halves' MMAs done
  const uint32_t tempty = tfull + 8u * 2;  // per accumulator: the eight fold warps read it
  const uint32_t drain = tempty + 8u * 2;  // two entries, one per issuing warp
  const uint32_t bready = drain + 8u * 2;  // the filter operand is built (eight fold warps)
  ptr += 8 * 23;
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(ptr);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ptr + 4);
  float* bias_s = reinterpret_cast<float*>(ptr + 8);  // per c (zero without bias)
  ptr += 8 + 8 * sizeof(float);
  if ((uint32_t)(ptr - c2i_smem) > dynamic_smem_bytes()) {  // same answer in every thread
    if (tid == 0) atomicExch(&g_c2i_err, DEV_ERR_LAYOUT);
    return;
  }

  if (tid == 0) {
    for (int s = 0; s < 4; ++s) {
      mbar_init(rfull + 8u * s, 1);  // the issuing thread's arrive + the copy's bytes
      mbar_init(rempty + 8u * s, 4);
      mbar_init(afull + 8u * s, 4);
      mbar_init(aempty + 8u * s, 2);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull + 8u * b, 2);
      mbar_init(tempty + 8u * b, 8);
    }
    mbar_init(drain, 1);
    mbar_init(drain + 8u, 1);
    mbar_init(bready, 8);
    *abort_flag = 0;
    for (int c = 0; c < 8; ++c)
      bias_s[c] = (p.bias != nullptr && c < p.C) ? static_cast<const float*>(p.bias)[c] : 0.f;
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

  // Stage it of this CTA = (tile blockIdx.x + (it / nkb) * gridDim.x, channel block it % nkb).
  const long long my_tiles = p.tiles > blockIdx.x ? (p.tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const long long nstage = my_tiles * p.nkb;
  const uint32_t chunk_bytes = (uint32_t)EH * 32u * 16u;  // one chunk of a staged operand

  if (warp < kMmaWarp) {
    // =============================================================== builders
    const int quarter = warp;
    const float* dy = static_cast<const float*>(p.dy);
    const long long PQ = (long long)p.P * p.Q;
    bool ok = true;
    int a = 0, slot = 0;              // operand slot and dy box slot of the current stage
    uint32_t aph = 0, rph = 0;        // their use parities
    for (long long t = blockIdx.x; t < p.tiles && ok; t += gridDim.x) {
      const Tile tc = tile_of(p, t);
      const int off = tc.q_lo - floor4(tc.q_lo);
      for (int kb = 0; kb < p.nkb; ++kb) {
        // (wait outcomes are made warp-uniform)
        if (!__all_sync(0xffffffffu, mbar_wait(aempty + 8u * a, aph ^ 1u, abort_flag, &g_c2i_err))) {
          ok = false;
          break;
        }
        if (p.use_tma &&
            !__all_sync(0xffffffffu, mbar_wait(rfull + 8u * slot, rph, abort_flag, &g_c2i_err))) {
          ok = false;
          break;
        }
        const uint32_t ast = a0 + (uint32_t)(a * p.a_bytes) + (uint32_t)lane * 16u;
        // staged dy rows p_lo - dlt_h + row, two at a time (more loads in flight)
        for (int row = quarter; row < EH; row += 8) {
          const bool two = row + 4 < EH;
          uint32_t v[2][kKS];
          if (p.use_tma) {
            const float* src = raw + (size_t)slot * (raw_bytes / 4) + row * 36 + lane + off;
#pragma unroll
            for (int k = 0; k < kKS; ++k) {
              v[0][k] = __float_as_uint(src[k * EH * 36]);
              v[1][k] = two ? __float_as_uint(src[k * EH * 36 + 4 * 36]) : 0u;
            }
          } else {
            const int q = tc.q_lo + lane;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int pp = tc.p_lo - p.dlt_h + row + 4 * u;
              const bool pv = (u == 0 || two) && pp >= 0 && pp < p.P && q >= 0 && q < p.Q;
              const float* src =
                  dy + (long long)tc.n * p.dy_nstride + (long long)kb * kKS * PQ + (long long)pp * p.Q + q;
#pragma unroll
              for (int k = 0; k < kKS; ++k)
                v[u][k] = (pv && kb * kKS + k < p.K) ? __float_as_uint(__ldg(src + (long long)k * PQ)) : 0u;
            }
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            if (u == 1 && !two) break;
            const uint32_t dst = ast + (uint32_t)((row + 4 * u) * 32 * 16);
#pragma unroll
            for (int j = 0; j < kKS / 4; ++j)
              st_shared_v4(dst + (uint32_t)j * chunk_bytes, v[u][4 * j], v[u][4 * j + 1], v[u][4 * j + 2],
                           v[u][4 * j + 3]);
          }
        }
        fence_proxy_async();  // this thread's operand writes, before the MMAs read them
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(afull + 8u * a);
          if (p.use_tma) mbar_arrive(rempty + 8u * slot);
        }
        if (++a == p.nast) {
          a = 0;
          aph ^= 1u;
        }
        if (p.use_tma && ++slot == p.nraw) {
          slot = 0;
          rph ^= 1u;
        }
      }
    }
  } else if (warp == kCopyWarp) {
    // =============================================================== dy tensor copies
    if (p.use_tma && lane == 0) {
      long long issued = 0, landed = 0;  // copies issued; copies whose slot was released after use
      bool ok = true;
      for (; issued < nstage; ++issued) {
        const int slot = (int)(issued % p.nraw);
        if (issued >= p.nraw) {  // the slot's previous stage read by all four builder warps
          if (!mbar_wait(rempty + 8u * slot, (uint32_t)(((issued / p.nraw) - 1) & 1), abort_flag, &g_c2i_err)) {
            ok = false;
            break;
          }
          landed = issued - p.nraw + 1;
          fence_proxy_async();
        }
        const Tile tc = tile_of(p, blockIdx.x + (issued / p.nkb) * gridDim.x);
        mbar_arrive_expect_tx(rfull + 8u * slot, (uint32_t)raw_bytes);
        tma_load_4d(raw0 + (uint32_t)(slot * raw_bytes), &p.tm_dy, floor4(tc.q_lo), tc.p_lo - p.dlt_h,
                    (int)(issued % p.nkb) * kKS, tc.n, rfull + 8u * slot);
      }
      // every copy is awaited before the CTA exits (released slots landed; wait for the rest)
      for (long long st = landed; st < issued; ++st)
        mbar_wait_drain(rfull + 8u * (uint32_t)(st % p.nraw), (uint32_t)((st / p.nraw) & 1));
      (void)ok;
    }
    __syncwarp();
  } else if (warp < kEpiWarp0) {
    // =============================================================== MMA issue
    const int mt = warp - kMmaWarp;  // 128-row half: anchor rows 4*mt .. 4*mt + 3
    const bool leader = elect_one();
    const uint32_t id = idesc(0, 128, p.Nr, 0, 0);
    const uint32_t bchunk = (uint32_t)p.Nr * 16u;
    const int nch = p.nkb * 4;
    int a = 0;
    uint32_t aph = 0;
    bool ok = __all_sync(0xffffffffu, mbar_wait(bready, 0u, abort_flag, &g_c2i_err));
    bool issued = false;
    long long tcount = 0;
    for (long long t = blockIdx.x; t < p.tiles && ok; t += gridDim.x, ++tcount) {
      const int buf = (int)(tcount & 1);
      if (!__all_sync(0xffffffffu, mbar_wait(tempty + 8u * buf, (uint32_t)(((tcount >> 1) & 1) ^ 1), abort_flag,
                                              &g_c2i_err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t dcol = tmem + (uint32_t)((buf * 2 + mt) * p.Nr);
      for (int kb = 0; kb < p.nkb; ++kb) {
        if (!__all_sync(0xffffffffu, mbar_wait(afull + 8u * a, aph, abort_flag, &g_c2i_err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (leader) {
          const uint32_t ast = a0 + (uint32_t)(a * p.a_bytes);
#pragma unroll 1
          for (int d = 0; d <= p.dlt_h; ++d) {
            // this half's anchor rows, moved back by d staged rows
            const uint32_t arow = ast + (uint32_t)((p.dlt_h + 4 * mt - d) * 32 * 16);
            const uint32_t bst = b0 + (uint32_t)(d * nch + kb * 4) * bchunk;
#pragma unroll
            for (int kk = 0; kk < kKS / 8; ++kk) {  // K = 8 channels (two chunks) per MMA
              const uint64_t ad = sdesc(arow + (uint32_t)(2 * kk) * chunk_bytes, chunk_bytes, 128u);
              const uint64_t bd = sdesc(bst + (uint32_t)(2 * kk) * bchunk, bchunk, 128u);
              mma_ss<0>(dcol, ad, bd, id, (kb | kk | d) != 0 ? 1u : 0u);
            }
          }
          tc_commit(aempty + 8u * a);
          if (kb == p.nkb - 1) tc_commit(tfull + 8u * buf);
        }
        __syncwarp();
        issued = true;
        if (++a == p.nast) {
          a = 0;
          aph ^= 1u;
        }
      }
      if (!ok) break;
    }
    if (!ok && issued && leader) {  // every MMA of this warp done before TMEM is released
      tc_commit(drain + 8u * (uint32_t)mt);
      mbar_wait_drain(drain + 8u * (uint32_t)mt, 0);
    }
    __syncwarp();
  } else {
    // =============================================================== fold and store
    const int ew = warp - kEpiWarp0;          // 0..7
    {
      // Filter operand, resident for the whole kernel (K-major), built while the first stages
      // are staged: for row shift d, chunk j (dy channels 4j..4j+3) and row n =
      // (c*sh + phi_h)*8 + s the filter tap (c, r, s) with r*dh = d*sh + phi_h; zero where no
      // such r < R exists, for padded s and rows, and past K.  Four rows per thread at a time,
      // all their loads issued before the first store.
      const float* w = static_cast<const float*>(p.w);
      const int nch = p.nkb * 4;
      const int nrows = (p.dlt_h + 1) * nch * p.Nr;
      const int et = tid - kEpiWarp0 * 32;
      for (int i0 = et; i0 < nrows; i0 += 4 * 256) {
        uint32_t v[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + 256 * u;
          v[u][0] = v[u][1] = v[u][2] = v[u][3] = 0u;
          if (i >= nrows) continue;
          const int dj = i / p.Nr, n = i - dj * p.Nr;
          const int d = dj / nch, j = dj - d * nch;
          const int cph = n >> 3, s = n & 7;
          const int c = cph / p.sh, phh = cph - c * p.sh;
          const int rd = d * p.sh + phh;  // r * dh
          const int r = rd / p.dh;
          if (c < p.C && s < p.S && rd % p.dh == 0 && r < p.R) {
            const int rr = p.flip ? p.R - 1 - r : r, ss = p.flip ? p.S - 1 - s : s;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int k = 4 * j + e;
              if (k < p.K) v[u][e] = __float_as_uint(__ldg(w + (((long long)k * p.C + c) * p.R + rr) * p.S + ss));
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (i0 + 256 * u < nrows)
            st_shared_v4(b0 + (uint32_t)(i0 + 256 * u) * 16u, v[u][0], v[u][1], v[u][2], v[u][3]);
      }
      fence_proxy_async();  // before the MMAs read the operand
      __syncwarp();
      if (lane == 0) mbar_arrive(bready);
    }
    const int quarter = warp & 3;             // the TMEM lane quarter this warp may read
    const int mt = ew >> 2;
    const int j = quarter + 4 * mt;           // anchor row of the tile
    uint32_t ctab[8];
#pragma unroll
    for (int phi = 0; phi < 8; ++phi) {
      uint32_t code = 0u;
      for (int s = 0; s < p.S; ++s) {
        const int d = s * p.dw - phi;
        if (phi < p.sw && d >= 0 && d % p.sw == 0) code |= (8u | (uint32_t)(d / p.sw)) << (4 * s);
      }
      ctab[phi] = code;
    }
    const int ngrp = p.C * p.sh;  // (c, phi_h) groups of 8 columns
    const long long HW = (long long)p.H * p.W;
    float* dx = static_cast<float*>(p.dx);
    const float beta = p.beta;
    const bool own = lane >= p.dlt_w;
    long long tcount = 0;
    for (long long t = blockIdx.x; t < p.tiles; t += gridDim.x, ++tcount) {
      const int buf = (int)(tcount & 1);
      if (!__all_sync(0xffffffffu,
                      mbar_wait(tfull + 8u * buf, (uint32_t)((tcount >> 1) & 1), abort_flag, &g_c2i_err)))
        break;
      tc_fence_after();
      const Tile tc = tile_of(p, t);
      const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)((buf * 2 + mt) * p.Nr);
      const int h0 = (tc.p_lo + j) * p.sh - p.ph;            // dx row of phase 0
      const int w0 = (tc.q_lo + lane) * p.sw - p.pw;         // dx column of phase 0
      float* dxn = dx + (long long)tc.n * p.dx_nstride;
      for (int g0 = 0; g0 < ngrp; g0 += kGB) {
        uint32_t z[kGB][8];
#pragma unroll
        for (int u = 0; u < kGB; ++u)
          if (g0 + u < ngrp) tmem_ld8(trow + (uint32_t)((g0 + u) * 8), z[u]);
        tmem_ld_wait();
        if (g0 + kGB >= ngrp) {  // this warp's TMEM reads of the tile are done
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty + 8u * buf);
        }
#pragma unroll
        for (int u = 0; u < kGB; ++u) {
          float out[8];
          fold_columns<SW, DW>(z[u], out, p.sw, ctab);
          const int g = g0 + u;
          if (g >= ngrp) continue;
          const int c = g / p.sh, phh = g - c * p.sh;
          const int h = h0 + phh;
          if (!own || h < 0 || h >= p.H) continue;
          float* orow = dxn + (long long)c * HW + (long long)h * p.W;
          const float bc = bias_s[c];
#pragma unroll
          for (int phi = 0; phi < 8; ++phi) {
            if (phi >= p.sw) break;
            const int wp = w0 + phi;
            if (wp < 0 || wp >= p.W) continue;
            float v = out[phi] + bc;
            if (beta != 0.f) v += beta * orow[wp];
            orow[wp] = v;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
  }
}

// ---------------------------------------------------------------------------- host side
size_t c2i_smem_bytes(const C2iPlan& p) {
  return 128 + (size_t)p.b_bytes + (size_t)p.nast * p.a_bytes + (size_t)p.nraw * (36 * p.EH * kKS * 4) + 8 * 23 + 8 +
         8 * sizeof(float);
}

static std::atomic<int> g_c2i_smem_set[4][kMaxDevices];

template <int SW, int DW>
static cudaError_t launch_c2i_t(const C2iPlan& p, unsigned grid, size_t smem, std::atomic<int>* set, cudaStream_t st) {
  const cudaError_t e = ensure_dyn_smem(dgrad_c2i_kernel<SW, DW>, smem, set);
  if (e != cudaSuccess) return e;
  dgrad_c2i_kernel<SW, DW><<<grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

// Column-fold variants with the stride and dilation as constants: (1, 1), (2, 1), (1, 2);
// any other pair runs the table-driven fold.
cudaError_t launch_c2i(const C2iPlan& p, int num_sms, cudaStream_t st) {
  const size_t smem = c2i_smem_bytes(p);
  const unsigned grid = (unsigned)std::max(1ll, std::min<long long>(p.tiles, (long long)num_sms));
  if (p.sw == 1 && p.dw == 1) return launch_c2i_t<1, 1>(p, grid, smem, g_c2i_smem_set[0], st);
  if (p.sw == 2 && p.dw == 1) return launch_c2i_t<2, 1>(p, grid, smem, g_c2i_smem_set[1], st);
  if (p.sw == 1 && p.dw == 2) return launch_c2i_t<1, 2>(p, grid, smem, g_c2i_smem_set[2], st);
  return launch_c2i_t<0, 0>(p, grid, smem, g_c2i_smem_set[3], st);
}

int c2i_take_error() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_c2i_err, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) cudaMemcpyToSymbol(g_c2i_err, &zero, sizeof(int));
  return v;
}

}  // namespace cg3

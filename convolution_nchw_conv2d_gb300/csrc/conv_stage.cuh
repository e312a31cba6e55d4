// conv_stage.cuh -- producer routines that stage NCHW activations into the shared-memory
// operand layouts of the tcgen05 kernels (see sm103_ptx.cuh for the layouts).
//
// Each routine is run by one producer group of 128 threads (4 warps) for one pipeline
// stage and only writes shared memory; the caller fences (fence.proxy.async) and arrives
// on the stage's mbarrier afterwards.  Global reads use 16-byte vector loads where the
// rows to be staged are contiguous and aligned in memory, and scalar loads otherwise;
// every element outside the source tensor is written as zero.  Work items are processed
// in batches: a thread issues all global loads of a batch before its first shared
// store, so several round trips to memory overlap.
#pragma once
#include <cstdint>
#include <type_traits>
#include <cuda_bf16.h>

#include "conv_plan.h"
#include "sm103_ptx.cuh"

namespace cg3 {

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}


__device__ __forceinline__ uint32_t comp(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// ------------------------------------------------------------------ pixel rows
// Source element offset of channel 0 of the pixel that plane `pl` of a TapPlan places at
// linear position L (L = n*EL*WL + e*WL + f; plane pixel (e, f) is source pixel
// (e*pl_step_h + pl_off_h, f*pl_step_w + pl_off_w)), or -1 outside the source tensor.
__device__ __forceinline__ int tap_src_offset(const TapPlan& p, uint32_t L, int pl) {
  if ((long long)L >= p.Mtot) return -1;
  const uint32_t n = fdiv(L, p.fd_img);
  const uint32_t rem = L - n * (uint32_t)p.fd_img.d;
  const uint32_t e = fdiv(rem, p.fd_WL);
  const int f = (int)(rem - e * (uint32_t)p.WL);
  const int h = (int)e * p.pl_step_h + p.pl_off_h[pl];
  const int w = f * p.pl_step_w + p.pl_off_w[pl];
  if (h < 0 || h >= p.Hs || w < 0 || w >= p.Ws) return -1;
  return (int)((long long)n * p.src_nstride + (long long)h * p.Ws + w);
}

// Layout [plane][chunk][row][16 bytes]: the 16 bytes of (plane, chunk j, row r) hold
// CHUNK consecutive channels cbase + j*CHUNK + e of the source pixel at linear position
// m0 + r of that plane (zero outside the tensor).
//
// Work item = (row, plane, group of G chunks): G*CHUNK = 16 scalar loads, one per channel,
// then G 16-byte shared stores.  Lanes take consecutive rows, so each load instruction
// of a warp reads consecutive pixels of one channel (coalesced wherever the rows are
// adjacent pixels) and each store instruction writes 512 contiguous bytes (no bank
// conflicts); no register transpose and no alignment condition.  Loads of the next item
// are issued before the stores of the current one.  Requires rows >= 128.
template <int DT>
__device__ __forceinline__ void stage_pixel_rows(const TapPlan& p, long long m0, uint32_t dst0, int cbase,
                                                 int nch, int gtid) {
  constexpr int CHUNK = DT == 0 ? 4 : 8;
  constexpr int G = 16 / CHUNK;  // chunks per item
  using E = typename std::conditional<DT == 0, uint32_t, uint16_t>::type;
  const E* src = static_cast<const E*>(p.src);
  const long long plane_stride = (long long)p.Hs * p.Ws;
  const int rows = p.rows, npl = p.npl;
  const int ngr = (nch + G - 1) / G;
  struct Item {
    int r, pl, jg;
  };
  auto load = [&](const Item& it, uint32_t (&v)[4 * G]) {
#pragma unroll
    for (int i = 0; i < 4 * G; ++i) v[i] = 0u;
    const int off = tap_src_offset(p, (uint32_t)(m0 + it.r), it.pl);
    if (off < 0) return;
    const int c0 = cbase + it.jg * G * CHUNK;
    const E* s0 = src + (long long)c0 * plane_stride + off;
    if (c0 + G * CHUNK <= p.Cs) {
#pragma unroll
      for (int e = 0; e < G * CHUNK; ++e) {
        const uint32_t x = (uint32_t)__ldg(s0 + e * plane_stride);
        if constexpr (DT == 0) v[e] = x;
        else v[e >> 1] |= x << (16 * (e & 1));
      }
    } else {
#pragma unroll
      for (int e = 0; e < G * CHUNK; ++e) {
        if (c0 + e >= p.Cs) break;
        const uint32_t x = (uint32_t)__ldg(s0 + e * plane_stride);
        if constexpr (DT == 0) v[e] = x;
        else v[e >> 1] |= x << (16 * (e & 1));
      }
    }
  };
  auto store = [&](const Item& it, const uint32_t (&v)[4 * G]) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int j = it.jg * G + g;
      if (j < nch)
        st_shared_v4(dst0 + (uint32_t)(((it.pl * nch + j) * rows + it.r) * 16), v[4 * g], v[4 * g + 1],
                     v[4 * g + 2], v[4 * g + 3]);
    }
  };
  // Items in [jg][pl][r] order, stride 128 (rows >= 128: one wrap per step at most).
  auto next = [&](Item& it) {
    it.r += 128;
    if (it.r >= rows) {
      it.r -= rows;
      if (++it.pl == npl) {
        it.pl = 0;
        ++it.jg;
      }
    }
  };
  Item a{gtid, 0, 0};
  uint32_t va[4 * G], vb[4 * G];
  if (a.jg < ngr) load(a, va);
  while (a.jg < ngr) {
    Item b = a;
    next(b);
    if (b.jg < ngr) load(b, vb);
    store(a, va);
    if (b.jg >= ngr) break;
    a = b;
    next(a);
    if (a.jg < ngr) load(a, va);
    store(b, vb);
  }
}

// ------------------------------------------------------------------ position rows
// Layout [chunk][row][16 bytes] with row = channel (or output channel) and the 16 bytes
// holding CHUNK consecutive positions: element (chunk j, row m, e) = src at channel
// mbase + m and position tab[CHUNK*j + e] (element offset of channel 0, -1 = zero).
// When a chunk's valid positions are a consecutive, aligned run from its start and
// `vec`, the chunk is one 16-byte cp.async per row (zero-filled past the run);
// otherwise scalar loads, batched.  Rows m >= mvalid are left untouched (the kernels
// never use them as data).
template <int DT>
__device__ __forceinline__ void stage_position_rows(const void* src_v, long long row_stride, const int* tab,
                                                    int nchunks, int nrows, int mvalid, uint32_t dst0,
                                                    int mbase, bool vec, int gtid) {
  constexpr int CHUNK = DT == 0 ? 4 : 8;
  constexpr int ESZ = DT == 0 ? 4 : 2;
  constexpr int U = 4;
  const int lane = gtid & 31, warp = gtid >> 5;
  const int mrows = mvalid < nrows ? mvalid : nrows;
  for (int j = warp; j < nchunks; j += 4) {
    const int o = tab[CHUNK * j];
    int nvalid = 0;
    bool contig = vec && o >= 0 && (o & (CHUNK - 1)) == 0;
#pragma unroll
    for (int e = 0; e < CHUNK; ++e) {
      const int oe = tab[CHUNK * j + e];
      if (oe >= 0 && oe == o + e && nvalid == e) ++nvalid;
      else if (oe >= 0) contig = false;  // a valid position that breaks the run
    }
    const uint32_t dbase = dst0 + (uint32_t)(j * nrows) * 16u;
    if (contig && nvalid > 0) {
      for (int m = lane; m < mrows; m += 32) {
        const char* s = static_cast<const char*>(src_v) + ((long long)(mbase + m) * row_stride + o) * ESZ;
        cp_async_16(dbase + (uint32_t)m * 16u, s, nvalid * ESZ);
      }
    } else {
      int offs[CHUNK];
#pragma unroll
      for (int e = 0; e < CHUNK; ++e) offs[e] = tab[CHUNK * j + e];
      for (int m0 = lane; m0 < mrows; m0 += 32 * U) {
        uint32_t w[U][4];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          w[u][0] = w[u][1] = w[u][2] = w[u][3] = 0u;
          const int m = m0 + 32 * u;
          if (m >= mrows) continue;
          const long long rb = (long long)(mbase + m) * row_stride;
#pragma unroll
          for (int e = 0; e < CHUNK; ++e) {
            if (offs[e] < 0) continue;
            if constexpr (DT == 0) {
              w[u][e] = __float_as_uint(__ldg(static_cast<const float*>(src_v) + rb + offs[e]));
            } else {
              w[u][e >> 1] |= (uint32_t)__ldg(static_cast<const uint16_t*>(src_v) + rb + offs[e]) << (16 * (e & 1));
            }
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int m = m0 + 32 * u;
          if (m < mrows) st_shared_v4(dbase + (uint32_t)m * 16u, w[u][0], w[u][1], w[u][2], w[u][3]);
        }
      }
    }
  }
}

}  // namespace cg3

namespace cg3 {

// 4-byte async copy global -> shared, zero-filled when !valid.
__device__ __forceinline__ void cp_async_4z(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0)
               : "memory");
}

}  // namespace cg3

namespace cg3 {

// ------------------------------------------------------------------ channel rows
// Layout [plane][row c][chunk j][16 bytes]: element (pl, c, CHUNK*j + e) = src at channel
// cbase + c (if < Cs) and position tab[pl*tabw + CHUNK*j + e] (element offset of channel 0,
// -1 = zero).  Rows hold positions contiguously.  A chunk whose positions are consecutive
// and 16-byte aligned in memory is one 16-byte cp.async; otherwise fp32 uses 4-byte
// cp.asyncs (zero-filled where invalid) and bf16 scalar loads.  The caller waits for
// cp.async before reading.
template <int DT>
__device__ __forceinline__ void stage_channel_rows(const void* src_v, long long plane_stride, int Cs,
                                                   const int* tab, int tabw, int npl, int nrows, int nchunks,
                                                   uint32_t dst0, int cbase, bool vec, int gtid) {
  constexpr int CHUNK = DT == 0 ? 4 : 8;
  constexpr int ESZ = DT == 0 ? 4 : 2;
  const int total = npl * nrows * nchunks;
  for (int it = gtid; it < total; it += 128) {
    const int j = it % nchunks;
    const int rc = it / nchunks;
    const int c = rc % nrows;
    const int pl = rc / nrows;
    const int* tt = tab + pl * tabw + CHUNK * j;
    const uint32_t d = dst0 + (uint32_t)it * 16u;
    const int cc = cbase + c;
    if (cc >= Cs) {
      st_shared_v4(d, 0u, 0u, 0u, 0u);
      continue;
    }
    const char* sc = static_cast<const char*>(src_v) + (long long)cc * plane_stride * ESZ;
    const int o = tt[0];
    bool contig = vec && o >= 0 && (o & (CHUNK - 1)) == 0;
    bool none = o < 0;
#pragma unroll
    for (int e = 1; e < CHUNK; ++e) {
      contig = contig && tt[e] == o + e;
      none = none && tt[e] < 0;
    }
    if (contig) {
      cp_async_16(d, sc + (long long)o * ESZ, 16);
    } else if (none) {
      st_shared_v4(d, 0u, 0u, 0u, 0u);
    } else if constexpr (DT == 0) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        cp_async_4z(d + 4u * e, tt[e] >= 0 ? (const void*)(sc + (long long)tt[e] * 4) : src_v, tt[e] >= 0);
    } else {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (tt[e] >= 0)
          w[e >> 1] |= (uint32_t)__ldg(reinterpret_cast<const uint16_t*>(sc) + tt[e]) << (16 * (e & 1));
      st_shared_v4(d, w[0], w[1], w[2], w[3]);
    }
  }
}

}  // namespace cg3

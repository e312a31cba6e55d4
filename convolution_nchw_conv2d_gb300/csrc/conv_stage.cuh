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

#include "sm103_ptx.cuh"

namespace cg3 {

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}


// 16-byte async copy global -> shared with zero fill beyond src_bytes (0..16).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}

// ------------------------------------------------------------------ pixel rows
// Layout [plane][chunk][row][16 bytes]: the 16 bytes of (plane, chunk j, row r) hold
// CHUNK consecutive channels cbase + j*CHUNK + e of the source pixel tab[plane][r]
// (the element offset of channel 0 of that pixel, -1 if outside the tensor).
//
// One staged row per thread: CHUNK scalar loads, one per channel, and one 16-byte shared
// store.  Lanes take consecutive rows, so each load instruction of a warp reads
// consecutive pixels of one channel (coalesced wherever the rows are adjacent pixels) and
// each store instruction writes 512 contiguous bytes (no bank conflicts); no register
// transpose and no alignment condition on the rows.  Requires rows >= 128.
template <int DT>
__device__ __forceinline__ void stage_pixel_rows(const void* src_v, long long plane_stride, int Cs,
                                                 const int* tab, int npl, int rows, uint32_t dst0,
                                                 int cbase, int nch, int gtid) {
  constexpr int CHUNK = DT == 0 ? 4 : 8;
  constexpr int U = DT == 0 ? 4 : 2;  // rows per batch: all loads of a batch precede its stores
  using E = typename std::conditional<DT == 0, uint32_t, uint16_t>::type;
  const E* src = static_cast<const E*>(src_v);
  // Item (plane pl, chunk j, row r), walked in [pl][j][r] order with stride 128.
  int pl = 0, j = 0, r = gtid;
  while (pl < npl) {
    uint32_t v[U][4];
    uint32_t dst[U];
    bool live[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      live[u] = pl < npl;
      v[u][0] = v[u][1] = v[u][2] = v[u][3] = 0u;
      dst[u] = dst0 + (uint32_t)(((pl * nch + j) * rows + r) * 16);
      if (live[u]) {
        const int off = tab[pl * rows + r];
        const int c0 = cbase + j * CHUNK;
        if (off >= 0) {
          const E* s0 = src + (long long)c0 * plane_stride + off;
          if (c0 + CHUNK <= Cs) {
#pragma unroll
            for (int e = 0; e < CHUNK; ++e) {
              const uint32_t x = (uint32_t)__ldg(s0 + e * plane_stride);
              if constexpr (DT == 0) v[u][e] = x;
              else v[u][e >> 1] |= x << (16 * (e & 1));
            }
          } else {
#pragma unroll
            for (int e = 0; e < CHUNK; ++e) {
              if (c0 + e >= Cs) break;
              const uint32_t x = (uint32_t)__ldg(s0 + e * plane_stride);
              if constexpr (DT == 0) v[u][e] = x;
              else v[u][e >> 1] |= x << (16 * (e & 1));
            }
          }
        }
      }
      r += 128;
      if (r >= rows) {
        r -= rows;
        if (++j == nch) {
          j = 0;
          ++pl;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (live[u]) st_shared_v4(dst[u], v[u][0], v[u][1], v[u][2], v[u][3]);
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

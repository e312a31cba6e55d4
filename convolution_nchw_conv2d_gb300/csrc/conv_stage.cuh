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
#include <cuda_bf16.h>

#include "sm103_ptx.cuh"

namespace cg3 {

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint4 ldg_v4(const void* p) { return __ldg(static_cast<const uint4*>(p)); }

__device__ __forceinline__ uint32_t comp(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
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
// Work item = CHUNK consecutive rows of one (plane, chunk), starting at row
// phase[plane] (mod CHUNK) when `vec`.  An item whose pixels are consecutive and
// CHUNK-aligned in memory is read with CHUNK 16-byte loads (one per channel) and
// transposed in registers; otherwise element by element.
template <int DT>
__device__ __forceinline__ void stage_pixel_rows(const void* src_v, long long plane_stride, int Cs,
                                                 const int* tab, int npl, int rows, uint32_t dst0,
                                                 int cbase, int nch, bool vec, const int* phase, int gtid) {
  constexpr int CHUNK = DT == 0 ? 4 : 8;
  constexpr int ESZ = DT == 0 ? 4 : 2;
  constexpr int U = DT == 0 ? 4 : 2;     // items per batch
  const int ngroups = rows / CHUNK + 2;  // covers every row for any phase in [0, CHUNK)
  const int total = npl * nch * ngroups;
  for (int base = gtid; base < total; base += 128 * U) {
    uint4 L[U][CHUNK];  // per item: one uint4 per channel holding CHUNK positions
    int r0s[U];
    uint32_t dbs[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int it = base + 128 * u;
#pragma unroll
      for (int c = 0; c < CHUNK; ++c) L[u][c] = make_uint4(0u, 0u, 0u, 0u);
      r0s[u] = -2 * CHUNK;  // no rows
      dbs[u] = 0u;
      if (it >= total) continue;
      const int pj = it / ngroups;
      const int g = it - pj * ngroups;
      const int pl = pj / nch;
      const int j = pj - pl * nch;
      const int c0 = cbase + j * CHUNK;
      const int nvc = Cs - c0;
      const int* t = tab + pl * rows;
      const int r0 = (vec ? phase[pl] : 0) - CHUNK + CHUNK * g;
      r0s[u] = r0;
      dbs[u] = dst0 + (uint32_t)(pj * rows) * 16u;
      bool contig = vec && r0 >= 0 && r0 + CHUNK <= rows && nvc >= CHUNK;
      const int o = contig ? t[r0] : -1;
      contig = contig && o >= 0 && (o & (CHUNK - 1)) == 0;
#pragma unroll
      for (int e = 1; e < CHUNK; ++e) contig = contig && (t[r0 + e] == o + e);
      if (contig) {
        const char* s = static_cast<const char*>(src_v) + ((long long)c0 * plane_stride + o) * ESZ;
#pragma unroll
        for (int c = 0; c < CHUNK; ++c) L[u][c] = ldg_v4(s + (long long)c * plane_stride * ESZ);
      } else {
#pragma unroll
        for (int e = 0; e < CHUNK; ++e) {
          const int r = r0 + e;
          const int oe = (r >= 0 && r < rows) ? t[r] : -1;
          if (oe < 0) continue;
#pragma unroll
          for (int c = 0; c < CHUNK; ++c) {
            if (c >= nvc) continue;
            uint32_t* w = reinterpret_cast<uint32_t*>(&L[u][c]);
            if constexpr (DT == 0) {
              w[e] = __float_as_uint(__ldg(static_cast<const float*>(src_v) + (long long)(c0 + c) * plane_stride + oe));
            } else {
              const uint32_t h = __ldg(static_cast<const uint16_t*>(src_v) + (long long)(c0 + c) * plane_stride + oe);
              w[e >> 1] |= h << (16 * (e & 1));
            }
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r0 = r0s[u];
#pragma unroll
      for (int q = 0; q < CHUNK; ++q) {
        const int r = r0 + q;
        if (r < 0 || r >= rows) continue;
        const uint32_t d = dbs[u] + (uint32_t)r * 16u;
        if constexpr (DT == 0) {
          st_shared_v4(d, comp(L[u][0], q), comp(L[u][1], q), comp(L[u][2], q), comp(L[u][3], q));
        } else {
          const uint32_t sel = (q & 1) ? 0x7632u : 0x5410u;
          const int i = q >> 1;
          st_shared_v4(d, __byte_perm(comp(L[u][0], i), comp(L[u][1], i), sel),
                       __byte_perm(comp(L[u][2], i), comp(L[u][3], i), sel),
                       __byte_perm(comp(L[u][4], i), comp(L[u][5], i), sel),
                       __byte_perm(comp(L[u][6], i), comp(L[u][7], i), sel));
        }
      }
    }
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

// ------------------------------------------------------------------ fp32 residue slots
// Layout [slot u][chunk j][row c][16 bytes]: element (u, j, c, e) = x at channel
// cbase + c and position tab[slot_plane[u]*rows + 4j + e + slot_res[u]] (element offset of
// channel 0, -1 = zero).  Used by the fp32 backward-filter, whose tf32 B operand must be
// K-major: each slot is one copy of an x plane shifted by a residue 0..3 so that every
// filter tap starts on a 16-byte chunk of some slot.  A chunk whose four positions are
// consecutive in memory is read with one or two aligned 16-byte loads.
__device__ __forceinline__ void stage_residue_rows_f32(const float* x, long long HW, int C, const int* tab,
                                                       int rows, int nsl, const int* slot_plane,
                                                       const int* slot_res, int nchunks, int NC, uint32_t dst0,
                                                       int cbase, bool vec, int gtid) {
  constexpr int U = 4;
  const int lane = gtid & 31, warp = gtid >> 5;
  const int cl = lane & 15, jj = lane >> 4;  // 16 channels x 2 chunks per warp instruction
  const int ncg = (NC + 15) >> 4;
  const int njp = (nchunks + 1) >> 1;
  const int per_slot = ncg * njp;
  const int total = nsl * per_slot;
  for (int base = warp; base < total; base += 4 * U) {
    uint32_t w[U][4];
    uint32_t dst[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      w[u][0] = w[u][1] = w[u][2] = w[u][3] = 0u;
      dst[u] = 0xFFFFFFFFu;
      const int it = base + 4 * u;
      if (it >= total) continue;
      const int us = it / per_slot;
      const int r = it - us * per_slot;
      const int cgi = r % ncg;
      const int jp = r / ncg;
      const int c = cgi * 16 + cl;
      const int j = jp * 2 + jj;
      if (c >= NC || j >= nchunks) continue;
      dst[u] = dst0 + (uint32_t)((us * nchunks + j) * NC + c) * 16u;
      const int cc = cbase + c;
      if (cc >= C) continue;
      const int* tt = tab + slot_plane[us] * rows + slot_res[us] + 4 * j;
      const int o = tt[0];
      const float* xc = x + (long long)cc * HW;
      const bool contig = vec && o >= 0 && tt[1] == o + 1 && tt[2] == o + 2 && tt[3] == o + 3;
      if (contig) {
        const int a = o & ~3;
        const uint4 v0 = ldg_v4(xc + a);
        const int d = o - a;
        if (d == 0) {
          w[u][0] = v0.x; w[u][1] = v0.y; w[u][2] = v0.z; w[u][3] = v0.w;
        } else {
          const uint4 v1 = ldg_v4(xc + a + 4);
          if (d == 1) { w[u][0] = v0.y; w[u][1] = v0.z; w[u][2] = v0.w; w[u][3] = v1.x; }
          else if (d == 2) { w[u][0] = v0.z; w[u][1] = v0.w; w[u][2] = v1.x; w[u][3] = v1.y; }
          else { w[u][0] = v0.w; w[u][1] = v1.x; w[u][2] = v1.y; w[u][3] = v1.z; }
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (tt[e] >= 0) w[u][e] = __float_as_uint(__ldg(xc + tt[e]));
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (dst[u] != 0xFFFFFFFFu) st_shared_v4(dst[u], w[u][0], w[u][1], w[u][2], w[u][3]);
  }
}

}  // namespace cg3

namespace cg3 {

// 4-byte async copy global -> shared, zero-filled when !valid.
__device__ __forceinline__ void cp_async_4z(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0)
               : "memory");
}

// ------------------------------------------------------------------ fp32 base copy (async)
// Layout [chunk j][row c][16 bytes]: element (j, c, e) = x at channel cbase + c and position
// tab[4j + e] (element offset of channel 0, -1 = zero).  Asynchronous: a chunk whose four
// positions are consecutive and 16-byte aligned in memory is one 16-byte cp.async per
// channel, a chunk with no valid position a zero-filling one, anything else four 4-byte
// cp.asyncs.  The caller waits (cp.async.wait_group) before reading.
__device__ __forceinline__ void stage_base_rows_async_f32(const float* x, long long HW, int C, const int* tab,
                                                          int nchunks, int NC, uint32_t dst0, int cbase,
                                                          bool vec, int gtid) {
  const int lane = gtid & 31, warp = gtid >> 5;
  for (int j = warp; j < nchunks; j += 4) {
    const int* tt = tab + 4 * j;
    const int o = tt[0];
    const bool none = o < 0 && tt[1] < 0 && tt[2] < 0 && tt[3] < 0;
    const bool contig = vec && o >= 0 && (o & 3) == 0 && tt[1] == o + 1 && tt[2] == o + 2 && tt[3] == o + 3;
    const uint32_t dbase = dst0 + (uint32_t)(j * NC) * 16u;
    for (int c = lane; c < NC; c += 32) {
      const int cc = cbase + c;
      const float* xc = x + (long long)(cc < C ? cc : 0) * HW;
      const uint32_t d = dbase + (uint32_t)c * 16u;
      if (cc >= C || none) {
        st_shared_v4(d, 0u, 0u, 0u, 0u);
      } else if (contig) {
        cp_async_16(d, xc + o, 16);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) cp_async_4z(d + 4u * e, tt[e] >= 0 ? xc + tt[e] : x, tt[e] >= 0);
      }
    }
  }
}

// Residue copy from the base copy, in shared memory: element (j, c, e) of the copy with
// residue r is element (j, c, e + r) of the base copy (carrying into chunk j + 1).
// The base copy must hold nchunks + 1 chunks.
__device__ __forceinline__ void stage_shift_rows_f32(uint32_t base0, uint32_t dst0, int r, int nchunks, int NC,
                                                     int gtid) {
  const int total = nchunks * NC;
  for (int i = gtid; i < total; i += 128) {
    const uint32_t s = base0 + (uint32_t)i * 16u;
    uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3) : "r"(s));
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3)
                 : "r"(s + (uint32_t)NC * 16u));
    uint32_t w0, w1, w2, w3;
    if (r == 1) { w0 = a1; w1 = a2; w2 = a3; w3 = b0; }
    else if (r == 2) { w0 = a2; w1 = a3; w2 = b0; w3 = b1; }
    else { w0 = a3; w1 = b0; w2 = b1; w3 = b2; }
    st_shared_v4(dst0 + (uint32_t)i * 16u, w0, w1, w2, w3);
  }
}

}  // namespace cg3

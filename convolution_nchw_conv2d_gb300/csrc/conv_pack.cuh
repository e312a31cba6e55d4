// conv_pack.cuh -- the operand packs shared by the kernel files: the channel-chunk pack of an
// NCHW activation (NhwcPackPlan) and the tap GEMM's filter pack (PackPlan), as per-unit device
// routines that a kernel of either file runs (alone, or two packs in one launch).
#pragma once
#include <cstdint>
#include <type_traits>
#include <cuda_bf16.h>

#include "conv_plan.h"
#include "sm103_ptx.cuh"

namespace cg3 {

__device__ __forceinline__ uint32_t comp4(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Shared memory of a channel-chunk pack unit: cg * CHUNK staged channel runs of ch_pitch elements.
inline size_t nhwc_pack_smem_bytes(const NhwcPackPlan& q, int dt) {
  return (size_t)q.cg * (dt == 0 ? 4 : 8) * q.ch_pitch * (dt == 0 ? 4 : 2);
}

// Staged position slot of position `pos` within a chunk's region of the transposed staging
// (CHUNK-aligned groups of CHUNK positions, the slot's low bits XORed with the group index:
// consecutive lanes storing the same position of consecutive groups hit different banks).
template <int CHUNK>
__device__ __forceinline__ int pack_slot(int pos) {
  return pos ^ ((pos / CHUNK) & (CHUNK - 1));
}

// Channel-chunk pack (NhwcPackPlan), work unit v, run by a whole block.  The unit's rows of
// its channel chunks are staged in shared memory, then every output 16-byte group (CHUNK
// channels of one plane position) is written, consecutive threads storing consecutive groups.
// Staging, when every channel row starts on a 16-byte boundary and W is a multiple of CHUNK:
// a thread loads a CHUNK x CHUNK block (one 16-byte load per channel: CHUNK consecutive
// positions), transposes it in registers (bf16: byte permutes of channel pairs) and stores
// CHUNK position-major 16-byte groups, so each output group is one 16-byte shared-memory read.
// Otherwise: channel runs by 16-byte asynchronous copies (or batched element loads) and each
// output group assembled from CHUNK shared-memory reads.  Channels past C are zero.
// `pk_smem` holds nhwc_pack_smem_bytes(p) bytes.
template <int DT>
__device__ __forceinline__ void nhwc_pack_unit(const NhwcPackPlan& p, uint32_t v, uint8_t* pk_smem) {
  constexpr int CHUNK = DT == 0 ? 4 : 8;
  constexpr int ESZ = DT == 0 ? 4 : 2;
  using E = typename std::conditional<DT == 0, uint32_t, uint16_t>::type;
  E* sm = reinterpret_cast<E*>(pk_smem);
  const uint32_t r = fdiv(v, p.fd_et);  // r = n * ngroups + group
  const int et = (int)(v - r * (uint32_t)p.n_etiles);
  const uint32_t n = fdiv(r, p.fd_ng);
  const int cc0 = (int)(r - n * (uint32_t)p.ngroups) * p.cg;
  const int ncc = min(p.cg, p.nchunk - cc0);
  const int e0 = et * p.te, ne = min(p.te, p.EX - e0);
  const int h_lo = e0 * p.step_h + p.off_h_min;
  const int h_hi = (e0 + ne - 1) * p.step_h + p.off_h_min + p.h_span;
  const int hl = max(h_lo, 0), hh = min(h_hi, p.H - 1);
  const int nr = hh - hl + 1;                          // staged rows (none when <= 0)
  const int nchs = min(ncc * CHUNK, p.C - cc0 * CHUNK);  // staged channels
  const long long HW = (long long)p.H * p.W;
  const E* base = static_cast<const E*>(p.src) + (long long)n * p.src_nstride + (long long)(cc0 * CHUNK) * HW +
                  (long long)(hl > 0 ? hl : 0) * p.W;
  const bool tr = (p.W % CHUNK) == 0 && ((reinterpret_cast<uintptr_t>(base) | (uintptr_t)(HW * ESZ)) & 15u) == 0;
  __syncthreads();  // the previous unit's reads of shared memory are done
  if (nr > 0) {
    const int len = nr * p.W;  // positions (elements per channel run)
    if (tr) {
      // transposed staging: chunk ccl's region holds ch_pitch 16-byte position slots
      const int nblk = len / CHUNK;
      const uint32_t s0 = smem_u32(sm);
      for (int i = (int)threadIdx.x; i < ncc * nblk; i += (int)blockDim.x) {
        const int ccl = i / nblk, b = i - ccl * nblk;
        uint4 x[CHUNK];
#pragma unroll
        for (int e = 0; e < CHUNK; ++e) {
          const int c = ccl * CHUNK + e;
          x[e] = c < nchs ? *reinterpret_cast<const uint4*>(base + (long long)c * HW + b * CHUNK)
                          : make_uint4(0u, 0u, 0u, 0u);
        }
        const uint32_t rb = s0 + (uint32_t)(ccl * p.ch_pitch) * 16u;
#pragma unroll
        for (int q = 0; q < CHUNK; ++q) {  // position b*CHUNK + q: CHUNK channels
          uint32_t o[4];
          if constexpr (DT == 0) {
            o[0] = comp4(x[0], q);
            o[1] = comp4(x[1], q);
            o[2] = comp4(x[2], q);
            o[3] = comp4(x[3], q);
          } else {
            const uint32_t sel = (q & 1) ? 0x7632u : 0x5410u;  // high or low halves of the pair
#pragma unroll
            for (int m = 0; m < 4; ++m) o[m] = __byte_perm(comp4(x[2 * m], q >> 1), comp4(x[2 * m + 1], q >> 1), sel);
          }
          const int slot = pack_slot<CHUNK>(b * CHUNK + q);
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(rb + (uint32_t)slot * 16u), "r"(o[0]),
                       "r"(o[1]), "r"(o[2]), "r"(o[3])
                       : "memory");
        }
      }
    } else {
      const bool vec = ((reinterpret_cast<uintptr_t>(base) | (uintptr_t)(HW * ESZ) | (uintptr_t)(len * ESZ)) & 15u) == 0;
      if (vec) {  // asynchronous 16-byte copies: all of a thread's copies in flight at once
        const int g = len * ESZ / 16;  // 16-byte groups per channel run
        const uint32_t s0 = smem_u32(sm);
        for (int i = (int)threadIdx.x; i < nchs * g; i += (int)blockDim.x) {
          const int c = i / g, k = i - c * g;
          cp_async_16(s0 + (uint32_t)((c * p.ch_pitch) * ESZ + k * 16), base + c * HW + k * (16 / ESZ), 16);
        }
        cp_async_commit();
        cp_async_wait<0>();
      } else {  // element loads, eight in flight per thread before their stores
        const int tot = nchs * len;
        for (int i0 = (int)threadIdx.x; i0 < tot; i0 += 8 * (int)blockDim.x) {
          E v8[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int i = i0 + q * (int)blockDim.x;
            if (i < tot) {
              const int c = i / len, k = i - c * len;
              v8[q] = base[c * HW + k];
            }
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int i = i0 + q * (int)blockDim.x;
            if (i < tot) {
              const int c = i / len, k = i - c * len;
              sm[c * p.ch_pitch + k] = v8[q];
            }
          }
        }
      }
    }
  }
  __syncthreads();
  // outputs (chunk ccl, plane pl, position gi of the unit's rows), flat index i; the (q, gi)
  // split advances incrementally (no division per output)
  const int groups = ne * p.WL;  // output groups per (chunk, plane)
  const int outs = ncc * p.npl * groups;
  int i = (int)threadIdx.x;
  int q = i / max(groups, 1), gi = i - q * groups;
  for (; i < outs; i += (int)blockDim.x) {
    const int ccl = q / p.npl, pl = q - ccl * p.npl;
    const int de = (int)fdiv((uint32_t)gi, p.fd_WL);
    const int f = gi - de * p.WL;
    const int h = (e0 + de) * p.step_h + p.off_h[pl];
    const int w = f * p.step_w + p.off_w[pl];
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (nr > 0 && h >= hl && h <= hh && w >= 0 && w < p.W) {
      const int pos = (h - hl) * p.W + w;
      if (tr) {
        uint32_t a, b2, c2, d2;
        const uint32_t addr =
            smem_u32(sm) + (uint32_t)(ccl * p.ch_pitch + pack_slot<CHUNK>(pos)) * 16u;
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(a), "=r"(b2), "=r"(c2), "=r"(d2) : "r"(addr));
        o = make_uint4(a, b2, c2, d2);
      } else {
        const int nch = min(CHUNK, nchs - ccl * CHUNK);
        const E* s0 = sm + (ccl * CHUNK) * p.ch_pitch + pos;
        uint32_t t[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int c = 0; c < CHUNK; ++c) {
          if (c < nch) {
            const uint32_t x = (uint32_t)s0[c * p.ch_pitch];
            if constexpr (DT == 0) t[c] = x;
            else t[c >> 1] |= x << (16 * (c & 1));
          }
        }
        o = make_uint4(t[0], t[1], t[2], t[3]);
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(p.dst) +
                 ((((long long)pl * p.nchunk + cc0 + ccl) * p.N + n) * p.EX + e0) * p.WL + gi;
    *dst = o;
    gi += (int)blockDim.x;
    while (gi >= groups) {
      gi -= groups;
      ++q;
    }
  }
}

// Filter pack for the tap GEMM, chunk idx (see PackPlan): wpack chunk index
// (((nt * nkb + kb) * ntaps + t) * NCH + j) * NT + n holds CHUNK consecutive source channels
// cs = kb*CB + j*CHUNK + e of out channel nt*NT + n for filter tap (tap_r[t], tap_s[t]); zero
// outside the tensor.  fp32 values are rounded to tf32 (round to nearest, ties away).  idx runs
// the tap index fastest, so the element reads of a warp fall on consecutive taps (r, s) of one
// filter row -- adjacent addresses of the KCRS filter -- and are coalesced; the 16-byte chunk
// stores are spread (one per tap slice) and merge in L2.
template <int DT>
__device__ __forceinline__ void pack_filter_one(const PackPlan& pp, uint32_t idx) {
  constexpr int ESZ = DT == 0 ? 4 : 2;
  constexpr int CHUNK = 16 / ESZ;
  using E = typename std::conditional<DT == 0, uint32_t, uint16_t>::type;
  const uint32_t NCH = (uint32_t)(pp.CB / CHUNK);
  const int RS = pp.R * pp.S;
  // 32-bit index arithmetic: the packed filter has fewer than 2^31 chunks (the planner keeps
  // it within its workspace cap)
  uint32_t rest = idx;
  const int t = (int)(rest % (uint32_t)pp.ntaps_total);
  rest /= (uint32_t)pp.ntaps_total;
  const int n = (int)(rest % (uint32_t)pp.NT);
  rest /= (uint32_t)pp.NT;
  const int j = (int)(rest % NCH);
  rest /= NCH;
  const int kb = (int)(rest % (uint32_t)pp.nkb);
  const int nt = (int)(rest / (uint32_t)pp.nkb);
  const int nn = nt * pp.NT + n;
  int r = pp.tap_r[t], s = pp.tap_s[t];
  if (pp.flip && r >= 0) {  // convolution mode: the filter rotated by 180 degrees
    r = pp.R - 1 - r;
    s = pp.S - 1 - s;
  }
  uint32_t out[4] = {0u, 0u, 0u, 0u};
  const int cs0 = kb * pp.CB + j * CHUNK;
  if (nn < pp.Cd && r >= 0 && pp.gd != 0) {  // block-diagonal: the group's slice of the filter
    const int g = nn / pp.gd, nl = nn - g * pp.gd;
    E v[CHUNK];
#pragma unroll
    for (int e = 0; e < CHUNK; ++e) {
      const int cs = cs0 + e;
      const bool in = cs < pp.Cs && cs / pp.gs == g;
      const long long idx = pp.transpose ? ((long long)cs * pp.C + nl) * RS : ((long long)nn * pp.C + (cs - g * pp.gs)) * RS;
      v[e] = in ? static_cast<const E*>(pp.w)[idx + r * pp.S + s] : (E)0;
    }
#pragma unroll
    for (int e = 0; e < CHUNK; ++e) {
      if constexpr (DT == 0) {
        uint32_t tf;
        asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(tf) : "f"(__uint_as_float(v[e])));
        out[e] = tf;
      } else {
        out[e >> 1] |= (uint32_t)v[e] << (16 * (e & 1));
      }
    }
  } else if (nn < pp.Cd && r >= 0) {
    const E* src = static_cast<const E*>(pp.w) +
                   (pp.transpose ? ((long long)cs0 * pp.C + nn) * RS : ((long long)nn * pp.C + cs0) * RS) + r * pp.S + s;
    const long long estep = pp.transpose ? (long long)pp.C * RS : RS;  // next source channel
    E v[CHUNK];
#pragma unroll
    for (int e = 0; e < CHUNK; ++e) v[e] = cs0 + e < pp.Cs ? src[e * estep] : (E)0;
#pragma unroll
    for (int e = 0; e < CHUNK; ++e) {
      if constexpr (DT == 0) {
        uint32_t tf;
        asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(tf) : "f"(__uint_as_float(v[e])));
        out[e] = tf;
      } else {
        out[e >> 1] |= (uint32_t)v[e] << (16 * (e & 1));
      }
    }
  }
  const long long oidx = (((long long)(nt * pp.nkb + kb) * pp.ntaps_total + t) * NCH + j) * pp.NT + n;
  reinterpret_cast<uint4*>(pp.wpack)[oidx] = make_uint4(out[0], out[1], out[2], out[3]);
}

}  // namespace cg3

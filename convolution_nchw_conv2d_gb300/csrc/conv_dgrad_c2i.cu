// conv_dgrad_c2i.cu -- backward-data (= deconvolution forward) for problems with few input
// channels C, where the tap GEMM's N dimension (C) would leave the tensor cores mostly idle.
//
// The backward-data sum in scatter form (page "LibMatrixCuDNNConvolutionAlgorithm.java", the
// backward-data algorithm and its descriptors; page "mkldnn_deconvolution.cc", the
// deconvolution forward that is the same operation): dy element (k, p, q) meets filter tap
// (c, r, s) once and lands on dx pixel (c, p*sh - ph + r*dh, q*sw - pw + s*dw).  So
//     Z[(p, q), (c, r, s)] = sum_k dy[k, p, q] * w[k, c, r, s]        (a GEMM, K deep)
//     dx[c, h, w]          = sum of Z[(p, q), (c, r, s)] over the (p, q, r, s) landing on (h, w).
//
// A tile stages 8 dy rows x 32 dy columns of positions (M = 256: two 128-row MMAs, one issuing
// warp each) with every dy channel, and the filter as B with N = C*R*8 rows ((c, r, s), s
// padded to 8), resident in shared memory; Z accumulates in TMEM (tf32 inputs, fp32 sums).
// The fold is exact and in a fixed order, in two steps:
//   columns: lane i of the warp that reads TMEM row j holds Z at dy position (j, i).  Output
//            column q*sw - pw + phi (phi < sw) receives tap s from position column
//            q - (s*dw - phi)/sw when s*dw - phi is a non-negative multiple of sw; a warp
//            shuffle brings those values to lane q, summed in ascending s, into the buffer
//            G[j][r][q*sw + phi] (one channel c at a time, two buffers alternating).
//   rows:    output row p*sh - ph + phi_h receives the row sums of tap r from dy row
//            p - (r*dh - phi_h)/sh under the same condition, summed in ascending r.
// Dy rows dlt_h..7 and columns dlt_w..31 of the tile are the ones whose pixels receive all
// their contributions from inside it (dlt = the largest shift); tiles step by the rest, so
// every dx pixel is written by exactly one tile, once (no atomics, no second pass).
//
// Roles: warps 0-3 stage dy (4-byte cp.async into the K-major operand layout, zero outside
// the tensor); warps 4-5 issue the MMAs; warps 6-13 fold and store.  Every wait is bounded.
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

constexpr int kStages = 3;
constexpr int kStageBytes = 8 * 256 * 16;  // 32 dy channels (8 chunks of 4) x 256 positions
constexpr int kThreads = 14 * 32;
constexpr int kMmaWarp = 4;                // warps 4 and 5: one 128-row half each
constexpr int kEpiWarp0 = 6;               // warps 6..13: fold and store
constexpr int kEpiThreads = 256;

// Each thread of the warp reads 8 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}

// Named barrier that also ORs a predicate over its members: every member gets the same answer.
__device__ __forceinline__ bool bar_any(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

struct Tile {
  int n, p_lo, q_lo;  // image; dy row and column of the tile's staged position (0, 0)
};

__device__ __forceinline__ Tile tile_of(const C2iPlan& p, long long t) {
  const long long per = (long long)p.ntp * p.ntq;
  Tile c;
  c.n = (int)(t / per);
  const int rem = (int)(t - (long long)c.n * per);
  const int tp = rem / p.ntq, tq = rem - tp * p.ntq;
  c.p_lo = p.p_start + tp * p.THp - p.dlt_h;
  c.q_lo = p.q_start + tq * p.TWq - p.dlt_w;
  return c;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1) dgrad_c2i_kernel(const __grid_constant__ C2iPlan p) {
  extern __shared__ __align__(16) uint8_t c2i_smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- shared memory: filter operand | dy stages | two fold buffers | row-fold table | barriers
  uint8_t* ptr = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(c2i_smem) + 127) & ~uintptr_t(127));
  const uint32_t b0 = smem_u32(ptr);
  ptr += p.b_bytes;
  const uint32_t a0 = smem_u32(ptr);
  ptr += kStages * kStageBytes;
  float* gbuf = reinterpret_cast<float*>(ptr);
  ptr += 2 * (size_t)p.g_floats * sizeof(float);
  int8_t* rtab = reinterpret_cast<int8_t*>(ptr);  // [phi_h][r]: dy row shift, or -1
  ptr += 256;
  const uint32_t full = smem_u32(ptr);
  const uint32_t empty = full + 8u * kStages;
  const uint32_t tfull = empty + 8u * kStages;
  const uint32_t tempty = tfull + 8u;
  const uint32_t drain = tempty + 8u;  // two entries, one per issuing warp
  ptr += 8 * (2 * kStages + 4);
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(ptr);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ptr + 4);
  ptr += 8;
  if ((uint32_t)(ptr - c2i_smem) > dynamic_smem_bytes()) {  // same answer in every thread
    if (tid == 0) atomicExch(&g_c2i_err, DEV_ERR_LAYOUT);
    return;
  }

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full + 8u * s, 128);  // every staging thread, after its own copies landed
      mbar_init(empty + 8u * s, 2);   // both issuing warps' commits
    }
    mbar_init(tfull, 2);
    mbar_init(tempty, 8);             // every fold warp, after its last TMEM read of the tile
    mbar_init(drain, 1);
    mbar_init(drain + 8u, 1);
    *abort_flag = 0;
    for (int ph = 0; ph < p.sh; ++ph)
      for (int r = 0; r < p.R; ++r) {
        const int d = r * p.dh - ph;
        rtab[ph * p.R + r] = (d >= 0 && d % p.sh == 0) ? (int8_t)(d / p.sh) : (int8_t)-1;
      }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32((const void*)tmem_holder), (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  {
    // Filter operand, resident for the whole kernel (K-major): chunk j = dy channels 4j..4j+3,
    // row n = (c*R + r)*8 + s; zero for padded s, padded rows and channels past K.
    const float* w = static_cast<const float*>(p.w);
    const int nrows = p.nkb * 8 * p.Npad;
    for (int i = tid; i < nrows; i += kThreads) {
      const int j = i / p.Npad, n = i - j * p.Npad;
      const int cr = n >> 3, s = n & 7;
      const int c = cr / p.R, r = cr - c * p.R;
      uint32_t v[4] = {0u, 0u, 0u, 0u};
      if (c < p.C && s < p.S) {
        const int rr = p.flip ? p.R - 1 - r : r, ss = p.flip ? p.S - 1 - s : s;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = 4 * j + e;
          if (k < p.K) v[e] = __float_as_uint(__ldg(w + (((long long)k * p.C + c) * p.R + rr) * p.S + ss));
        }
      }
      st_shared_v4(b0 + (uint32_t)i * 16u, v[0], v[1], v[2], v[3]);
    }
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp < kMmaWarp) {
    // =============================================================== staging
    // Operand layout [chunk j][row m][16 B], m = dy row (0..7) * 32 + dy column (0..31).  One
    // copy instruction covers 8 rows x 4 channels of one chunk: lane = row (lane / 4) and
    // channel (lane % 4), so the warp reads four 32-byte runs and writes 128 contiguous bytes.
    const float* dy = static_cast<const float*>(p.dy);
    const long long PQ = (long long)p.P * p.Q;
    const int e = lane & 3, sub = lane >> 2;
    long long it = 0;
    bool ok = true;
    for (long long t = blockIdx.x; t < p.tiles && ok; t += gridDim.x) {
      const Tile tc = tile_of(p, t);
      const float* dyn = dy + (long long)tc.n * p.dy_nstride;
      uint32_t colv = 0u, rowv = 0u;
#pragma unroll
      for (int ib = 0; ib < 4; ++ib) {
        const int q = tc.q_lo + 8 * ib + sub;
        if (q >= 0 && q < p.Q) colv |= 1u << ib;
      }
#pragma unroll
      for (int pr = 0; pr < 8; ++pr) {
        const int pp = tc.p_lo + pr;
        if (pp >= 0 && pp < p.P) rowv |= 1u << pr;
      }
      const long long pos0 = (long long)tc.p_lo * p.Q + tc.q_lo + sub;
      for (int kb = 0; kb < p.nkb; ++kb, ++it) {
        const int s = (int)(it % kStages);
        const uint32_t ph = (uint32_t)((it / kStages) & 1);
        if (!mbar_wait(empty + 8u * s, ph ^ 1u, abort_flag, &g_c2i_err)) {
          ok = false;
          break;
        }
        const uint32_t st = a0 + (uint32_t)s * kStageBytes;
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const int j = 2 * warp + jj;
          const int k = kb * 32 + 4 * j + e;
          const bool kv = k < p.K;
          const long long kofs = (long long)k * PQ + pos0;
          const uint32_t dj = st + (uint32_t)j * 4096u + (uint32_t)sub * 16u + (uint32_t)e * 4u;
#pragma unroll
          for (int pr = 0; pr < 8; ++pr) {
#pragma unroll
            for (int ib = 0; ib < 4; ++ib) {
              const bool v = kv && ((rowv >> pr) & 1u) && ((colv >> ib) & 1u);
              const float* src = v ? dyn + kofs + (long long)pr * p.Q + 8 * ib : dy;
              cp_async_4(dj + (uint32_t)(pr * 512 + ib * 128), src, v);
            }
          }
        }
        cp_async_commit();
        if (it > 0) {  // the previous stage's copies of this thread have landed
          cp_async_wait<1>();
          fence_proxy_async();
          mbar_arrive(full + 8u * (uint32_t)((it - 1) % kStages));
        }
      }
    }
    cp_async_wait<0>();
    if (ok && it > 0) {
      fence_proxy_async();
      mbar_arrive(full + 8u * (uint32_t)((it - 1) % kStages));
    }
  } else if (warp < kEpiWarp0) {
    // =============================================================== MMA issue
    const int mt = warp - kMmaWarp;  // 128-row half of the tile
    const bool leader = elect_one();
    const uint32_t id = idesc(0, 128, p.Npad, 0, 0);
    const uint32_t dcol = tmem + (uint32_t)(mt * p.Npad);
    const uint32_t bchunk = (uint32_t)p.Npad * 16u;
    long long it = 0;
    uint32_t tph = 0;
    bool ok = true, issued = false;
    for (long long t = blockIdx.x; t < p.tiles; t += gridDim.x) {
      if (!mbar_wait(tempty, tph ^ 1u, abort_flag, &g_c2i_err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int kb = 0; kb < p.nkb; ++kb, ++it) {
        const int s = (int)(it % kStages);
        const uint32_t ph = (uint32_t)((it / kStages) & 1);
        if (!mbar_wait(full + 8u * s, ph, abort_flag, &g_c2i_err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (leader) {
          const uint32_t ast = a0 + (uint32_t)s * kStageBytes + (uint32_t)mt * 2048u;
          const uint32_t bst = b0 + (uint32_t)(kb * 8) * bchunk;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // K = 8 (two chunks) per MMA
            const uint64_t ad = sdesc(ast + (uint32_t)kk * 8192u, 4096u, 128u);
            const uint64_t bd = sdesc(bst + (uint32_t)(2 * kk) * bchunk, bchunk, 128u);
            mma_ss<0>(dcol, ad, bd, id, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(empty + 8u * s);
          if (kb == p.nkb - 1) tc_commit(tfull);
        }
        __syncwarp();
        issued = true;
      }
      if (!ok) break;
      tph ^= 1u;
    }
    if (!ok && issued && leader) {  // every MMA of this warp done before TMEM is released
      tc_commit(drain + 8u * (uint32_t)mt);
      mbar_wait_drain(drain + 8u * (uint32_t)mt, 0);
    }
    __syncwarp();
  } else {
    // =============================================================== fold and store
    const int ew = warp - kEpiWarp0;          // 0..7
    const int quarter = warp & 3;             // the TMEM lane quarter this warp may read
    const int j = quarter + 4 * (ew >> 2);    // tile dy row = TMEM row group of this warp
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)((ew >> 2) * p.Npad);
    // Column fold per output column phase phi: 4 bits per tap s (bit 3: s lands on phi,
    // bits 0-2: the lane shift (s*dw - phi)/sw).
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
    const int GW = 32 * p.sw;
    const int TH = p.THp * p.sh, TW = p.TWq * p.sw;
    const long long HW = (long long)p.H * p.W;
    const float* bias = static_cast<const float*>(p.bias);
    float* dx = static_cast<float*>(p.dx);
    uint32_t tph = 0, u = 0;
    for (long long t = blockIdx.x; t < p.tiles; t += gridDim.x) {
      const bool okw = mbar_wait(tfull, tph, abort_flag, &g_c2i_err);
      if (bar_any(1, kEpiThreads, !okw)) break;
      tc_fence_after();
      const Tile tc = tile_of(p, t);
      const int h_base = (tc.p_lo + p.dlt_h) * p.sh - p.ph;
      const int w_base = (tc.q_lo + p.dlt_w) * p.sw - p.pw;
      float* dxn = dx + (long long)tc.n * p.dx_nstride;
      for (int c = 0; c < p.C; ++c, ++u) {
        float* G = gbuf + (size_t)(u & 1u) * p.g_floats;
        // ---- columns: G[j][r][lane*sw + phi]
        for (int r0 = 0; r0 < p.R; r0 += 4) {
          uint32_t z[4][8];
#pragma unroll
          for (int uu = 0; uu < 4; ++uu)
            if (r0 + uu < p.R) tmem_ld8(trow + (uint32_t)((c * p.R + r0 + uu) * 8), z[uu]);
          tmem_ld_wait();
#pragma unroll
          for (int uu = 0; uu < 4; ++uu) {
            if (r0 + uu >= p.R) break;
            float* grow = G + (size_t)(j * p.R + r0 + uu) * GW + lane * p.sw;
#pragma unroll
            for (int phi = 0; phi < 8; ++phi) {
              if (phi >= p.sw) break;
              float acc = 0.f;
#pragma unroll
              for (int s = 0; s < 8; ++s) {
                const uint32_t code = (ctab[phi] >> (4 * s)) & 15u;
                if (code & 8u) acc += __shfl_up_sync(0xffffffffu, __uint_as_float(z[uu][s]), code & 7u);
              }
              grow[phi] = acc;
            }
          }
        }
        if (c == p.C - 1) {  // this warp's TMEM reads of the tile are done
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty);
        }
        named_bar_sync(1, kEpiThreads);
        // ---- rows, epilogue and store: the tile's owned dx rows, one row per warp at a time
        const float bc = bias != nullptr ? __ldg(bias + c) : 0.f;
        float* dxc = dxn + (long long)c * HW;
        for (int hr = ew; hr < TH; hr += 8) {
          const int h = h_base + hr;
          if (h < 0 || h >= p.H) continue;
          const int hq = hr / p.sh;
          const int prow0 = p.dlt_h + hq, phh = hr - hq * p.sh;
          const int8_t* rt = rtab + phh * p.R;
          for (int wc = lane; wc < TW; wc += 32) {
            const int wp = w_base + wc;
            if (wp < 0 || wp >= p.W) continue;
            const int col = p.dlt_w * p.sw + wc;
            float acc = 0.f;
            for (int r = 0; r < p.R; ++r) {
              const int d = rt[r];
              if (d >= 0) acc += G[(size_t)((prow0 - d) * p.R + r) * GW + col];
            }
            float* o = dxc + (long long)h * p.W + wp;
            float v = acc + bc;
            if (p.beta != 0.f) v += p.beta * *o;
            *o = v;
          }
        }
      }
      tph ^= 1u;
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
  return 128 + (size_t)p.b_bytes + (size_t)kStages * kStageBytes + 2 * (size_t)p.g_floats * sizeof(float) + 256 +
         8 * (2 * kStages + 4) + 8;
}

static std::atomic<int> g_c2i_smem_set[kMaxDevices];

cudaError_t launch_c2i(const C2iPlan& p, int num_sms, cudaStream_t st) {
  const size_t smem = c2i_smem_bytes(p);
  const cudaError_t e = ensure_dyn_smem(dgrad_c2i_kernel, smem, g_c2i_smem_set);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)std::max(1ll, std::min<long long>(p.tiles, (long long)num_sms));
  dgrad_c2i_kernel<<<grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

int c2i_take_error() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_c2i_err, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) cudaMemcpyToSymbol(g_c2i_err, &zero, sizeof(int));
  return v;
}

}  // namespace cg3

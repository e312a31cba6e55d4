// conv_wgrad.cu -- backward-filter convolution on sm_103a tensor cores.
//
//   dw[k,c,r,s] = sum_{n,p,q} X(n, c, p*sh - ph + r, q*sw - pw + s) * dy[n,k,p,q]
// (the filter gradient of the cuDNN backward-filter call in Apache SystemDS
// LibMatrixCuDNNConvolutionAlgorithm.java; deconvolution's backward-weights in
// Apache MXNet mkldnn_deconvolution.cc is the same product with the weight's roles
// swapped).  The reduction runs over the forward linear position space L (see
// conv_plan.h): dy is zero at positions with no output, and tap (r,s) reads the x
// phase plane of (r mod sh, s mod sw) at L + tap_off.
//
// One CTA tile = 128 output channels k x NC input channels c x a group of taps x one
// range of positions (split-K).  Per pipeline stage (KB positions):
//   producers (warps 0-7, two groups taking stages in turn) stage dy[k, L] K-major and
//     x in the core-matrix layout:
//     bf16 as an MN-major operand (channels along chunks, positions along rows, a
//     tap is a row offset); fp32 as K-major copies per (plane, offset mod 4), since
//     tf32 operands must be K-major (an MN-major tf32 B reads as zeros);
//   the MMA lane copies each 128 x 32-byte dy slice into TMEM with tcgen05.cp and
//     issues one tcgen05.mma per tap with A from TMEM and B = x at the tap's row
//     offset, so dy is read from shared memory once for all taps;
//   epilogue warps (8-11) write each tap's 128 x NC fp32 partial sums.
// A second kernel adds the split partials in a fixed order (deterministic) and
// writes dw in KCRS, rounding to bf16 for bf16 tensors.
#include "conv_plan.h"
#include "conv_stage.cuh"
#include "sm103_ptx.cuh"

namespace cg3 {

__device__ int g_wgrad_err;

namespace {
// CTA roles: warps 0-7 two producer groups taking pipeline stages in turn, warps 8-11
// epilogue, warp 12 TMEM allocation + tcgen05.cp / tcgen05.mma issue.
constexpr int kThreads = 416;
constexpr int kProdThreads = 128;
constexpr int kEpiWarp0 = 8;
constexpr int kMmaWarp = 12;
constexpr int kAbufCols = 32;  // 4 TMEM staging buffers of 8 columns for dy slices

__device__ __forceinline__ uint32_t bar_at(uint32_t base, int i) { return base + 8u * (uint32_t)i; }

struct WTile {
  int kt, ct, tg, sp;
};
__device__ __forceinline__ WTile decode_wtile(const WgradPlan& p, long long t) {
  WTile w;
  w.kt = (int)(t % p.n_ktiles);
  long long r = t / p.n_ktiles;
  w.ct = (int)(r % p.n_ctiles);
  r /= p.n_ctiles;
  w.tg = (int)(r % p.n_tgroups);
  w.sp = (int)(r / p.n_tgroups);
  return w;
}
}  // namespace

template <int DT>
__global__ void __launch_bounds__(kThreads, 1) wgrad_kernel(const __grid_constant__ WgradPlan p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  constexpr int ESZ = DT == 0 ? 4 : 2;
  constexpr int CHUNK = 16 / ESZ;
  constexpr int KIND = DT;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int S = p.stages;
  const int rows = p.rows;
  const int KB = p.KB;
  const int NCA = KB / CHUNK;     // dy chunks per stage
  const int NCB = p.NC / CHUNK;   // bf16: x chunks per plane per stage

  uint8_t* ptr = smem_raw;
  const uint32_t a0 = smem_u32(ptr);
  ptr += (size_t)S * p.a_stage_bytes;
  const uint32_t b0 = smem_u32(ptr);
  ptr += (size_t)S * p.b_stage_bytes;
  const int tab_ints = KB + p.npl * rows;
  int* tabs = reinterpret_cast<int*>(ptr);  // one table set per producer group
  ptr += (size_t)2 * tab_ints * sizeof(int);
  // Per plan tap: start of its B operand relative to the stage base, in 16-byte units.
  uint32_t* tapb = reinterpret_cast<uint32_t*>(ptr);
  ptr += (size_t)p.ntaps * sizeof(uint32_t);
  ptr = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ptr) + 15) & ~uintptr_t(15));
  const uint32_t full = smem_u32(ptr);
  const uint32_t empty = full + 8u * S;
  const uint32_t accf = empty + 8u * S;
  const uint32_t acce = accf + 8u;
  const uint32_t drain = acce + 8u;
  ptr += 8 * (2 * S + 3);
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(ptr);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ptr + 4);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_at(full, s), kProdThreads);
      mbar_init(bar_at(empty, s), 1);
    }
    mbar_init(accf, 1);
    mbar_init(acce, 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32((const void*)tmem_holder), (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  for (int g = 0; g < p.n_tgroups; ++g)
    for (int t = p.tg_begin[g] + tid; t < p.tg_begin[g] + p.tg_count[g]; t += kThreads) {
      if constexpr (DT == 0)
        tapb[t] = (uint32_t)(((p.tap_slot[t] - p.tg_slot_begin[g]) * p.slot_chunks + p.tap_q[t]) * p.NC);
      else
        tapb[t] = (uint32_t)(p.tap_plane[t] * NCB * rows + p.tap_off[t]);
    }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const long long img = (long long)p.EL * p.WL;
  const long long HW = (long long)p.H * p.W;
  const long long PQ = (long long)p.P * p.Q;

  if (warp < kEpiWarp0) {
    // =============================================================== producers
    const int grp = warp >> 2;
    const int gtid = tid & (kProdThreads - 1);
    int* dytab = tabs + grp * tab_ints;
    int* xtab = dytab + KB;
    long long counter = 0;
    bool ok = true;
    for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
      const WTile wt = decode_wtile(p, t);
      const long long lbeg = (long long)wt.sp * p.split_len;
      long long lend = lbeg + p.split_len;
      if (lend > p.Mtot) lend = p.Mtot;
      const int kbase = wt.kt * 128;
      const int cbase = wt.ct * p.NC;
      const long long xbase = DT == 0 ? 4ll * p.tg_qmin[wt.tg] - p.x_shift : 0ll;
      const int sl0 = p.tg_slot_begin[wt.tg];
      const int nsl = p.tg_nslots[wt.tg];
      for (long long l0 = lbeg; l0 < lend; l0 += KB, ++counter) {
        // Stage ownership is a pure function of the counter, so all threads of a group
        // pass the same named barriers even after an abort (which only skips work).
        if ((int)(counter & 1) != grp) continue;
        const int stage = (int)(counter % S);
        const uint32_t ephase = (uint32_t)((counter / S) & 1);
        // Position tables for this stage (this group's own copy).
        named_bar_sync(1 + grp, kProdThreads);
        for (int i = gtid; i < tab_ints; i += kProdThreads) {
          if (i < KB) {
            const long long L = l0 + i;
            int off = -1;
            if (L < lend) {
              const int n = (int)(L / img);
              const int rem = (int)(L - (long long)n * img);
              const int e = rem / p.WL;
              const int f = rem - e * p.WL;
              if (e < p.P && f < p.Q) off = (int)((long long)n * p.K * PQ + (long long)e * p.Q + f);
            }
            dytab[i] = off;
          } else {
            const int j = i - KB;
            const int pl = j / rows;
            const int row = j - pl * rows;
            const long long L = l0 + xbase + row;
            int off = -1;
            if (L >= 0 && L < p.Mtot) {
              const int n = (int)(L / img);
              const int rem = (int)(L - (long long)n * img);
              const int e = rem / p.WL;
              const int f = rem - e * p.WL;
              const int h = e * p.pl_step_h + p.pl_off_h[pl];
              const int w = f * p.pl_step_w + p.pl_off_w[pl];
              if (h >= 0 && h < p.H && w >= 0 && w < p.W)
                off = (int)((long long)n * p.C * HW + (long long)h * p.W + w);
            }
            xtab[j] = off;
          }
        }
        named_bar_sync(1 + grp, kProdThreads);
        if (!ok) continue;
        if (!mbar_wait(bar_at(empty, stage), ephase ^ 1u, abort_flag, &g_wgrad_err)) {
          ok = false;
          continue;
        }
        const uint32_t a_st = a0 + (uint32_t)stage * p.a_stage_bytes;
        const uint32_t b_st = b0 + (uint32_t)stage * p.b_stage_bytes;
        // dy: [chunk][k row][CHUNK positions], rows k >= K left as they are (never used).
        stage_position_rows<DT>(p.dy, PQ, dytab, NCA, 128, p.K - kbase, a_st, kbase, p.vec_dy != 0, gtid);
        if constexpr (DT == 0) {
          // Residue-0 copy of each plane asynchronously, then (once every thread's copies
          // have landed) the shifted residue copies from it, in shared memory.
          const uint32_t slot_bytes = (uint32_t)(p.slot_chunks * p.NC) * 16u;
          for (int u = 0; u < nsl; ++u)
            if (p.slot_res[sl0 + u] == 0)
              stage_base_rows_async_f32(static_cast<const float*>(p.x), HW, p.C, xtab + p.slot_plane[sl0 + u] * rows,
                                        p.slot_chunks, p.NC, b_st + (uint32_t)u * slot_bytes, cbase, p.vec_x != 0,
                                        gtid);
          cp_async_wait<0>();
          named_bar_sync(1 + grp, kProdThreads);
          for (int u = 0; u < nsl; ++u) {
            const int r = p.slot_res[sl0 + u];
            if (r != 0)
              stage_shift_rows_f32(b_st + (uint32_t)(p.slot_base[sl0 + u] - sl0) * slot_bytes,
                                   b_st + (uint32_t)u * slot_bytes, r, p.nchunks, p.NC, gtid);
          }
        } else {
          stage_pixel_rows<DT>(p.x, HW, p.C, xtab, p.npl, rows, b_st, cbase, NCB, p.vec_x != 0, p.vec_phase,
                               gtid);
          cp_async_wait<0>();
        }
        fence_proxy_async();
        mbar_arrive(bar_at(full, stage));
      }
    }
    cp_async_wait<0>();
  } else if (warp < kMmaWarp) {
    // =============================================================== epilogue
    const int q = warp & 3;
    uint32_t aphase = 0;
    for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
      const WTile wt = decode_wtile(p, t);
      if (!mbar_wait(accf, aphase, abort_flag, &g_wgrad_err)) break;
      tc_fence_after();
      const int k = wt.kt * 128 + q * 32 + lane;
      const int tap0 = p.tg_begin[wt.tg];
      const int ntg = p.tg_count[wt.tg];
      for (int ti = 0; ti < ntg; ++ti) {
        float* dst = p.partial + ((long long)wt.sp * p.ntaps + p.tap_id[tap0 + ti]) * p.c_pad * (long long)p.k_pad;
        const uint32_t tcol = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(kAbufCols + ti * p.NC);
        for (int c0 = 0; c0 < p.NC; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(tcol + (uint32_t)c0, r);
          tmem_ld_wait();
          if (k < p.K) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int c = wt.ct * p.NC + c0 + j;
              if (c < p.C) dst[(long long)c * p.k_pad + k] = __uint_as_float(r[j]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce);
      aphase ^= 1u;
    }
  } else {
    // =============================================================== MMA issuer
    if (lane == 0) {
      const uint32_t id = idesc(KIND, 128, p.NC, 0, DT == 0 ? 0 : 1);
      long long counter = 0;
      uint32_t aphase = 0;
      int abuf = 0;
      bool ok = true;
      bool issued_any = false;
      const int KSTEP = 2 * CHUNK;  // positions per MMA
      for (long long t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
        const WTile wt = decode_wtile(p, t);
        const long long lbeg = (long long)wt.sp * p.split_len;
        long long lend = lbeg + p.split_len;
        if (lend > p.Mtot) lend = p.Mtot;
        const int tap0 = p.tg_begin[wt.tg];
        const int ntg = p.tg_count[wt.tg];
        if (!mbar_wait(acce, aphase ^ 1u, abort_flag, &g_wgrad_err)) break;
        tc_fence_after();
        bool first = true;
        for (long long l0 = lbeg; l0 < lend; l0 += KB, ++counter) {
          const int stage = (int)(counter % S);
          const uint32_t fphase = (uint32_t)((counter / S) & 1);
          if (!mbar_wait(bar_at(full, stage), fphase, abort_flag, &g_wgrad_err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_st = a0 + (uint32_t)stage * p.a_stage_bytes;
          const uint32_t b_st = b0 + (uint32_t)stage * p.b_stage_bytes;
          // fp32: K-major x slot copies (chunk stride NC*16); bf16: MN-major x planes
          // (positions along rows).  Per k-step the B start moves by 2 chunks / KSTEP rows.
          const uint64_t bdesc0 = DT == 0 ? sdesc(b_st, (uint32_t)p.NC * 16u, 128u)
                                          : sdesc(b_st, 128u, (uint32_t)rows * 16u);
          const uint32_t b_lo0 = (uint32_t)bdesc0, b_hi = (uint32_t)(bdesc0 >> 32);
          const uint32_t b_ks = DT == 0 ? 2u * (uint32_t)p.NC : (uint32_t)KSTEP;
          const uint64_t cdesc0 = sdesc(a_st, 128u * 16u, 128u);
          for (int ks = 0; ks < NCA / 2; ++ks) {
            const uint32_t a_tm = tmem + (uint32_t)(abuf * 8);
            tmem_cp_128x256b(a_tm, cdesc0 + (uint32_t)(2 * ks * 128));
            if (++abuf == kAbufCols / 8) abuf = 0;
            const uint32_t acc_in = first ? 0u : 1u;
            const uint32_t blo = b_lo0 + (uint32_t)ks * b_ks;
            uint32_t dcol = tmem + (uint32_t)kAbufCols;
            for (int ti = 0; ti < ntg; ++ti) {
              mma_ts_lh<KIND>(dcol, a_tm, blo + tapb[tap0 + ti], b_hi, id, acc_in);
              dcol += (uint32_t)p.NC;
            }
            first = false;
          }
          tc_commit(bar_at(empty, stage));
          issued_any = true;
        }
        if (!ok) break;
        tc_commit(accf);
        aphase ^= 1u;
      }
      if (!ok && issued_any) {
        tc_commit(drain);
        mbar_wait_drain(drain, 0);
      }
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

size_t wgrad_smem_bytes(const WgradPlan& p) {
  size_t b = (size_t)p.stages * (p.a_stage_bytes + p.b_stage_bytes);
  b += (size_t)2 * (p.KB + p.npl * p.rows) * sizeof(int) + (size_t)p.ntaps * sizeof(uint32_t);
  b = (b + 15) & ~size_t(15);
  b += 8 * (2 * p.stages + 3) + 16;
  return b + 1024;
}

cudaError_t launch_wgrad(const WgradPlan& p, int dt, int grid, cudaStream_t st) {
  const size_t smem = wgrad_smem_bytes(p);
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

// conv_wgrad.cu -- backward-filter convolution on sm_103a tensor cores.
//
//   dw[k,c,r,s] = sum_{n,p,q} X(n, c, p*sh - ph + r, q*sw - pw + s) * dy[n,k,p,q]
// (the filter gradient of the cuDNN backward-filter call in Apache SystemDS
// LibMatrixCuDNNConvolutionAlgorithm.java; deconvolution's backward-weights in Apache
// MXNet mkldnn_deconvolution.cc is the same product with the weight's roles swapped).
//
// One GEMM per tile (see WgradPlan in conv_plan.h): rows m = (c, tap) of the filter,
// columns = output channels k, reduction over the forward linear position space L.
// Per pipeline stage (KB positions) the producers stage dy[k, L] (K-major, positions
// contiguous) and the few x channels the tile's rows need; builder warps then write the
// im2col rows A[(c, tap), L] = X_plane(tap)[c, L + tap_off] straight into TMEM
// (tcgen05.st), one k-step at a time, and one thread issues tcgen05.mma with A from TMEM
// and B = dy from shared memory (kind::tf32 / kind::f16 with bf16), accumulating the
// 128 x NK tile in TMEM.  The builders then store the tile's fp32 partial sums, with
// 16-byte stores along k.  A second kernel adds the split partials in a fixed order
// (deterministic) and writes dw in KCRS, rounding to bf16 for bf16 tensors.
#include "conv_plan.h"
#include "conv_stage.cuh"
#include "sm103_ptx.cuh"

namespace cg3 {

__device__ int g_wgrad_err;

namespace {
// CTA roles (544 threads): warps 0-7 two producer groups taking pipeline stages in turn
// (cp.async of the dy tile and the x tile), warps 8-15 two builder sets (set h builds the
// im2col A operand of every k-step with k-step mod 2 == h into TMEM, and runs half of the
// epilogue), warp 16 TMEM allocation + MMA issue.
constexpr int kThreads = 544;
constexpr int kProdThreads = 128;
constexpr int kBuildWarp0 = 8;
constexpr int kMmaWarp = 16;
constexpr int kNabuf = 4;  // TMEM A buffers (8 columns each)

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
}  // namespace

template <int DT>
__global__ void __launch_bounds__(kThreads, 1) wgrad_kernel(const __grid_constant__ WgradPlan p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  constexpr int ESZ = DT == 0 ? 4 : 2;
  constexpr int CHUNK = 16 / ESZ;
  constexpr int KSTEP = 2 * CHUNK;  // positions per MMA
  constexpr int KIND = DT;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int S = p.stages;
  const int KB = p.KB;
  const int nks = KB / KSTEP;  // k-steps per stage (even)
  const int xrow = p.xrow;  // staged x positions per row

  uint8_t* ptr = smem_raw;
  const uint32_t a0 = smem_u32(ptr);  // dy tiles
  ptr += (size_t)S * p.a_stage_bytes;
  const uint32_t b0 = smem_u32(ptr);  // x tiles
  ptr += (size_t)S * p.b_stage_bytes;
  const int tab_ints = KB + p.npl * xrow;
  int* tabs = reinterpret_cast<int*>(ptr);  // one table set per producer group
  ptr += (size_t)2 * tab_ints * sizeof(int);
  ptr = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ptr) + 15) & ~uintptr_t(15));
  const uint32_t full = smem_u32(ptr);
  const uint32_t empty = full + 8u * S;
  const uint32_t afull = empty + 8u * S;
  const uint32_t aempty = afull + 8u * kNabuf;
  const uint32_t accf = aempty + 8u * kNabuf;
  const uint32_t acce = accf + 8u;
  const uint32_t drain = acce + 8u;
  ptr += 8 * (2 * S + 2 * kNabuf + 3);
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
    mbar_init(accf, 1);
    mbar_init(acce, 8);
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
  const uint32_t dcol0 = tmem + (uint32_t)(kNabuf * 8);  // accumulator columns

  const long long HW = (long long)p.H * p.W;
  const long long PQ = (long long)p.P * p.Q;

  if (warp < kBuildWarp0) {
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
      const int kbase = wt.nt * p.NK;
      const int cbase = (wt.mt * 128) / p.RS;
      for (long long l0 = lbeg; l0 < lend; l0 += KB, ++counter) {
        // Stage ownership is a pure function of the counter, so all threads of a group
        // pass the same named barriers even after an abort (which only skips work).
        if ((int)(counter & 1) != grp) continue;
        const int stage = (int)(counter % S);
        const uint32_t ephase = (uint32_t)((counter / S) & 1);
        named_bar_sync(1 + grp, kProdThreads);
        for (int i = gtid; i < tab_ints; i += kProdThreads) {
          if (i < KB) {
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
          } else {
            const int j = i - KB;
            const int pl = j / xrow;
            const int xi = j - pl * xrow;
            const long long L = l0 - p.x_shift + xi;
            int off = -1;
            if (L >= 0 && L < p.Mtot) {
              const uint32_t n = fdiv((uint32_t)L, p.fd_img);
              const uint32_t rem = (uint32_t)L - n * p.fd_img.d;
              const int e = (int)fdiv(rem, p.fd_WL);
              const int f = (int)rem - e * p.WL;
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
        // dy: [chunk][k row][CHUNK positions]; x: [plane][channel][positions]
        stage_position_rows<DT>(p.dy, PQ, dytab, KB / CHUNK, p.NK, p.K - kbase, a_st, kbase, p.vec_dy != 0, gtid);
        stage_channel_rows<DT>(p.x, HW, p.C, xtab, xrow, p.npl, p.xch, p.xchunks, b_st, cbase, p.vec_x != 0, gtid);
        cp_async_commit();  // wait_group only covers committed groups
        cp_async_wait<0>();
        fence_proxy_async();
        mbar_arrive(bar_at(full, stage));
      }
    }
    cp_async_commit();
    cp_async_wait<0>();
  } else if (warp < kMmaWarp) {
    // =============================================================== builders + epilogue
    const int set = (warp - kBuildWarp0) >> 2;  // builds k-steps with index mod 2 == set
    const int q = warp & 3;                      // TMEM lane quarter
    long long counter = 0, kglob = 0;
    uint32_t aphase = 0;
    bool ok = true;
    for (long long t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
      const WTile wt = decode_wtile(p, t);
      const long long lbeg = (long long)wt.sp * p.split_len;
      long long lend = lbeg + p.split_len;
      if (lend > p.Mtot) lend = p.Mtot;
      const int cbase = (wt.mt * 128) / p.RS;
      const int m = wt.mt * 128 + q * 32 + lane;  // this thread's A row (c, tap)
      const bool mvalid = m < p.M;
      const int c = mvalid ? m / p.RS : 0;
      const int tap = mvalid ? m - c * p.RS : 0;
      // byte offset of this row's first needed x element inside a stage's x tile
      const uint32_t xoff =
          (uint32_t)(((p.tap_plane[tap] * p.xch + (c - cbase)) * xrow + p.tap_off[tap] + p.x_shift) * ESZ);
      for (long long l0 = lbeg; l0 < lend && ok; l0 += KB, ++counter) {
        const int stage = (int)(counter % S);
        const uint32_t fphase = (uint32_t)((counter / S) & 1);
        if (!mbar_wait(bar_at(full, stage), fphase, abort_flag, &g_wgrad_err)) {
          ok = false;
          break;
        }
        const uint32_t xs = b0 + (uint32_t)stage * p.b_stage_bytes + xoff;
        for (int ks = 0; ks < nks; ++ks, ++kglob) {
          if ((ks & 1) != set) continue;
          const int abuf = (int)(kglob % kNabuf);
          const uint32_t use = (uint32_t)((kglob / kNabuf) & 1);
          if (!mbar_wait(bar_at(aempty, abuf), use ^ 1u, abort_flag, &g_wgrad_err)) {
            ok = false;
            break;
          }
          uint32_t v[8];
          if (mvalid) {
            const uint32_t a = xs + (uint32_t)(ks * KSTEP * ESZ);
            if constexpr (DT == 0) {
#pragma unroll
              for (int e = 0; e < 8; ++e)
                asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v[e]) : "r"(a + 4u * e));
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                uint16_t lo, hi;
                asm volatile("ld.shared.u16 %0, [%1];" : "=h"(lo) : "r"(a + 4u * e));
                asm volatile("ld.shared.u16 %0, [%1];" : "=h"(hi) : "r"(a + 4u * e + 2u));
                v[e] = (uint32_t)lo | ((uint32_t)hi << 16);
              }
            }
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0u;
          }
          tc_fence_after();
          tmem_st8(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(abuf * 8), v);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_at(afull, abuf));
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_at(empty, stage));  // done reading this stage's x tile
      }
      if (!ok) break;
      // ---- epilogue: this set writes half of the accumulator columns
      if (!mbar_wait(accf, aphase, abort_flag, &g_wgrad_err)) break;
      tc_fence_after();
      const int tapo = tap;  // filter tap index r*S + s
      const int half = p.NK >> 1;
      const int k0 = wt.nt * p.NK + set * half;
      float* dst = p.partial + (((long long)wt.sp * p.RS + tapo) * p.C + c) * (long long)p.K;
      for (int c0 = 0; c0 < half; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(dcol0 + ((uint32_t)(q * 32) << 16) + (uint32_t)(set * half + c0), r);
        tmem_ld_wait();
        if (mvalid) {
          const int kk = k0 + c0;
          if (kk + 16 <= p.K && ((p.K & 3) == 0)) {
#pragma unroll
            for (int j = 0; j < 16; j += 4)
              *reinterpret_cast<uint4*>(dst + kk + j) = make_uint4(r[j], r[j + 1], r[j + 2], r[j + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (kk + j < p.K) dst[kk + j] = __uint_as_float(r[j]);
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
      const uint32_t id = idesc(KIND, 128, p.NK, 0, 0);
      const uint32_t b_hi = (uint32_t)(sdesc(0u, 0u, 128u) >> 32);
      long long counter = 0, kglob = 0;
      uint32_t aphase = 0;
      bool ok = true;
      bool issued_any = false;
      for (long long t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
        const WTile wt = decode_wtile(p, t);
        const long long lbeg = (long long)wt.sp * p.split_len;
        long long lend = lbeg + p.split_len;
        if (lend > p.Mtot) lend = p.Mtot;
        if (!mbar_wait(acce, aphase ^ 1u, abort_flag, &g_wgrad_err)) break;
        tc_fence_after();
        bool first = true;
        for (long long l0 = lbeg; l0 < lend && ok; l0 += KB, ++counter) {
          const int stage = (int)(counter % S);
          const uint32_t fphase = (uint32_t)((counter / S) & 1);
          if (!mbar_wait(bar_at(full, stage), fphase, abort_flag, &g_wgrad_err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // B = dy tile, K-major [chunk][k row][16 B]: k-step ks uses chunks 2ks, 2ks+1.
          uint32_t blo = (uint32_t)sdesc(a0 + (uint32_t)stage * p.a_stage_bytes, (uint32_t)p.NK * 16u, 0u);
          const uint32_t b_ks = 2u * (uint32_t)p.NK;
          for (int ks = 0; ks < nks; ++ks, ++kglob) {
            const int abuf = (int)(kglob % kNabuf);
            const uint32_t use = (uint32_t)((kglob / kNabuf) & 1);
            if (!mbar_wait(bar_at(afull, abuf), use, abort_flag, &g_wgrad_err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            mma_ts_lh<KIND>(dcol0, tmem + (uint32_t)(abuf * 8), blo, b_hi, id, first ? 0u : 1u);
            tc_commit(bar_at(aempty, abuf));
            issued_any = true;
            first = false;
            blo += b_ks;
          }
          if (!ok) break;
          tc_commit(bar_at(empty, stage));
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
  b += (size_t)2 * (p.KB + p.npl * p.xrow) * sizeof(int);
  b = (b + 15) & ~size_t(15);
  b += 8 * (2 * p.stages + 2 * 4 + 3) + 16;
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

// conv_tap_gemm.cu -- forward and backward-data convolution on sm_103a tensor cores.
//
// Both ops are the same implicit GEMM (see conv_plan.h):
//   D[position L, out_channel n] = sum_{tap t} sum_{source channel c}
//        S_plane(t)[c, L + tap_off[t]] * Wpack[t][n][c]
// Forward: S = x split into stride phase planes, n = K output channel, every tap
// (r,s) of the filter (Apache SystemDS LibMatrixCuDNNConvolutionAlgorithm.java:
// NCHW x, KCRS w, cross-correlation).  Backward-data: S = dy, n = C input channel,
// the output dx is split into stride phases and each phase gathers only the taps
// that reach it, with the filter read as (K, C) transposed and the taps reversed;
// this is deconvolution forward with the weight's in/out roles swapped (Apache
// MXNet mkldnn_deconvolution.cc, MKLDNNDeconvFwd::Execute comment).
//
// CTA roles (288 threads, persistent over tiles):
//   warps 0-3  producers: stage source rows for CB channels into shared memory in
//              the core-matrix interleaved layout (fp32: 4-byte cp.async with zero
//              fill; bf16: register gather), and bulk-copy the packed filter slice.
//   warps 4-7  epilogue: TMEM -> registers -> NCHW global stores, coalesced along
//              output positions; bf16 outputs rounded to nearest even.
//   warp 8     TMEM allocation; lane 0 issues tcgen05.mma (kind::tf32 for fp32,
//              kind::f16 with bf16 operands) accumulating in TMEM.
#include <mutex>
#include <vector>

#include "conv_plan.h"
#include "sm103_ptx.cuh"

namespace cg3 {

__device__ int g_tap_err;

namespace {

constexpr int kThreads = 288;
constexpr int kProdThreads = 128;

struct TapSmem {
  uint32_t a0, b0;       // stage region bases (shared addresses)
  int* rowtab;
  uint32_t full, bfull, empty, accf, acce, drain;  // barrier arrays (shared addresses)
};

__device__ __forceinline__ uint32_t bar_at(uint32_t base, int i) { return base + 8u * (uint32_t)i; }

struct TileCoord {
  int ph, mt, nt;
};

__device__ __forceinline__ TileCoord decode_tile(const TapPlan& p, long long t) {
  TileCoord c;
  c.nt = (int)(t % p.n_ntiles);
  long long rest = t / p.n_ntiles;
  c.mt = (int)(rest % p.n_mtiles);
  c.ph = (int)(rest / p.n_mtiles);
  return c;
}

template <int DT>
__device__ __forceinline__ void store_out(void* dst, long long idx, uint32_t bits) {
  if constexpr (DT == 0) {
    static_cast<float*>(dst)[idx] = __uint_as_float(bits);
  } else {
    static_cast<__nv_bfloat16*>(dst)[idx] = __float2bfloat16_rn(__uint_as_float(bits));
  }
}

}  // namespace

template <int DT>
__global__ void __launch_bounds__(kThreads, 1) tap_gemm_kernel(const __grid_constant__ TapPlan p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  constexpr int ESZ = DT == 0 ? 4 : 2;
  constexpr int CHUNK = 16 / ESZ;  // elements per 16-byte chunk
  constexpr int KIND = DT;         // 0: tf32, 1: f16-kind with bf16

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int S = p.stages;
  const int NCH = p.CB / CHUNK;
  const int rows = p.rows;

  // ---- shared memory carve-up
  uint8_t* ptr = smem_raw;
  TapSmem sm;
  sm.a0 = smem_u32(ptr);
  ptr += (size_t)S * p.a_stage_bytes;
  sm.b0 = smem_u32(ptr);
  ptr += (size_t)S * p.b_stage_bytes;
  sm.rowtab = reinterpret_cast<int*>(ptr);
  ptr += (size_t)p.npl * rows * sizeof(int);
  ptr = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ptr) + 15) & ~uintptr_t(15));
  uint64_t* bars = reinterpret_cast<uint64_t*>(ptr);
  sm.full = smem_u32(bars);
  sm.bfull = sm.full + 8u * S;
  sm.empty = sm.bfull + 8u * S;
  sm.accf = sm.empty + 8u * S;
  sm.acce = sm.accf + 16u;
  sm.drain = sm.acce + 16u;
  ptr += 8 * (3 * S + 5);
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(ptr);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ptr + 4);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_at(sm.full, s), kProdThreads);
      mbar_init(bar_at(sm.bfull, s), 1);
      mbar_init(bar_at(sm.empty, s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_at(sm.accf, a), 1);
      mbar_init(bar_at(sm.acce, a), 4);
    }
    mbar_init(sm.drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(smem_u32((const void*)tmem_holder), (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const long long img = (long long)p.EL * p.WL;
  const long long HsWs = (long long)p.Hs * p.Ws;
  const long long HdWd = (long long)p.Hd * p.Wd;
  const int MT = 128 * p.MH;
  const int b_tap_bytes = NCH * p.NT * 16;

  if (warp < 4) {
    // =============================================================== producers
    const int ptid = tid;
    int stage = 0;
    uint32_t ephase = 0;
    int pending = -1;  // fp32: stage whose cp.async group is still in flight
    bool ok = true;
    // Per stage slot: parity of the last bulk copy issued into it (for the exit drain).
    uint32_t issued_mask = 0, issued_par = 0;
    for (long long t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
      const TileCoord tc = decode_tile(p, t);
      const int ntaps = p.ph_ntaps[tc.ph];
      if (ntaps == 0) continue;
      const long long m0 = (long long)tc.mt * MT;
      // Row table: source offset (channel 0) of every staged row of every plane.
      named_bar_sync(1, kProdThreads);
      for (int i = ptid; i < p.npl * rows; i += kProdThreads) {
        const int pl = i / rows;
        const int row = i - pl * rows;
        const long long L = m0 + row;
        int off = -1;
        if (L < p.Mtot) {
          const int n = (int)(L / img);
          const int rem = (int)(L - (long long)n * img);
          const int e = rem / p.WL;
          const int f = rem - e * p.WL;
          const int h = e * p.pl_step_h + p.pl_off_h[pl];
          const int w = f * p.pl_step_w + p.pl_off_w[pl];
          if (h >= 0 && h < p.Hs && w >= 0 && w < p.Ws)
            off = (int)((long long)n * p.Cs * HsWs + (long long)h * p.Ws + w);
        }
        sm.rowtab[i] = off;
      }
      named_bar_sync(1, kProdThreads);
      for (int kb = 0; kb < p.nkb; ++kb) {
        if (!mbar_wait(bar_at(sm.empty, stage), ephase ^ 1u, abort_flag, &g_tap_err)) {
          ok = false;
          break;
        }
        const uint32_t a_st = sm.a0 + (uint32_t)stage * p.a_stage_bytes;
        const uint32_t b_st = sm.b0 + (uint32_t)stage * p.b_stage_bytes;
        if (ptid == 0) {
          const uint32_t bytes = (uint32_t)(ntaps * b_tap_bytes);
          const long long img_off =
              ((long long)(tc.nt * p.nkb + kb) * p.ntaps_total + p.ph_tap_begin[tc.ph]) * b_tap_bytes;
          mbar_arrive_expect_tx(bar_at(sm.bfull, stage), bytes);
          bulk_g2s(b_st, static_cast<const uint8_t*>(p.wpack) + img_off, bytes, bar_at(sm.bfull, stage));
          issued_mask |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (ephase << stage);
        }
        const int cbase = kb * p.CB;
        if constexpr (DT == 0) {
          // fp32: lane = (row within 8, channel within chunk); one warp instruction
          // fills 8 rows x 16 bytes = 128 contiguous bytes.
          const float* src = static_cast<const float*>(p.src);
          const int c4 = lane & 3;
          const int rsub = lane >> 2;
          for (int pj = 0; pj < p.npl * NCH; ++pj) {
            const int pl = pj / NCH;
            const int j = pj - pl * NCH;
            const int cs = cbase + j * 4 + c4;
            const bool cv = cs < p.Cs;
            const float* gc = src + (long long)(cv ? cs : 0) * HsWs;
            const uint32_t dbase = a_st + (uint32_t)(pj * rows) * 16u + (uint32_t)c4 * 4u;
            const int* tab = sm.rowtab + pl * rows;
#pragma unroll 4
            for (int row = warp * 8 + rsub; row < rows; row += 32) {
              const int off = tab[row];
              const bool v = cv && off >= 0;
              cp_async_4(dbase + (uint32_t)row * 16u, v ? gc + off : src, v);
            }
          }
          cp_async_commit();
          if (pending >= 0) {
            cp_async_wait<1>();
            fence_proxy_async();
            mbar_arrive(bar_at(sm.full, pending));
          }
          pending = stage;
        } else {
          // bf16: one thread gathers 8 channels of one row and writes one 16-byte chunk.
          const uint16_t* src = static_cast<const uint16_t*>(p.src);
          for (int pj = 0; pj < p.npl * NCH; ++pj) {
            const int pl = pj / NCH;
            const int j = pj - pl * NCH;
            const int c0 = cbase + j * 8;
            const int nv = min(8, p.Cs - c0);
            const uint16_t* gc = src + (long long)(nv > 0 ? c0 : 0) * HsWs;
            const int* tab = sm.rowtab + pl * rows;
            const uint32_t dbase = a_st + (uint32_t)(pj * rows) * 16u;
#pragma unroll 2
            for (int row = ptid; row < rows; row += kProdThreads) {
              const int off = tab[row];
              uint32_t wv[4] = {0u, 0u, 0u, 0u};
              if (off >= 0) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  if (e < nv) {
                    const uint32_t v = __ldg(gc + off + (long long)e * HsWs);
                    wv[e >> 1] |= v << (16 * (e & 1));
                  }
                }
              }
              asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dbase + (uint32_t)row * 16u),
                           "r"(wv[0]), "r"(wv[1]), "r"(wv[2]), "r"(wv[3])
                           : "memory");
            }
          }
          fence_proxy_async();
          mbar_arrive(bar_at(sm.full, stage));
        }
        if (++stage == S) {
          stage = 0;
          ephase ^= 1u;
        }
      }
    }
    if constexpr (DT == 0) {
      cp_async_wait<0>();
      if (pending >= 0 && ok) {
        fence_proxy_async();
        mbar_arrive(bar_at(sm.full, pending));
      }
    }
    // Drain: never leave a bulk copy in flight into shared memory that is about to be
    // released.  In a normal run every one of these has long completed.
    if (ptid == 0) {
      for (int s = 0; s < S; ++s) {
        if (issued_mask & (1u << s)) {
          mbar_wait_drain(bar_at(sm.bfull, s), (issued_par >> s) & 1u);
        }
      }
    }
  } else if (warp < 8) {
    // =============================================================== epilogue
    const int q = warp & 3;
    int acc = 0;
    uint32_t aphase = 0;
    for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
      const TileCoord tc = decode_tile(p, t);
      const int ntaps = p.ph_ntaps[tc.ph];
      const long long m0 = (long long)tc.mt * MT;
      if (ntaps != 0) {
        if (!mbar_wait(bar_at(sm.accf, acc), aphase, abort_flag, &g_tap_err)) break;
        tc_fence_after();
      }
      for (int h = 0; h < p.MH; ++h) {
        const int m = h * 128 + q * 32 + lane;
        const long long L = m0 + m;
        bool valid = false;
        long long obase = 0;
        if (L < p.Mtot) {
          const int n = (int)(L / img);
          const int rem = (int)(L - (long long)n * img);
          const int e = rem / p.WL;
          const int f = rem - e * p.WL;
          const int oh = e * p.ph_step_h + p.ph_off_h[tc.ph];
          const int ow = f * p.ph_step_w + p.ph_off_w[tc.ph];
          valid = oh >= 0 && oh < p.Hd && ow >= 0 && ow < p.Wd;
          obase = (long long)n * p.Cd * HdWd + (long long)oh * p.Wd + ow;
        }
        for (int c0 = 0; c0 < p.NT; c0 += 16) {
          uint32_t r[16];
          if (ntaps != 0) {
            tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)((acc * p.MH + h) * p.NT + c0), r);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = 0u;
          }
          if (valid) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int nn = tc.nt * p.NT + c0 + j;
              if (nn < p.Cd) store_out<DT>(p.dst, obase + (long long)nn * HdWd, r[j]);
            }
          }
        }
      }
      if (ntaps != 0) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_at(sm.acce, acc));
        if (++acc == p.ACCB) {
          acc = 0;
          aphase ^= 1u;
        }
      }
    }
  } else {
    // =============================================================== MMA issuer
    if (lane == 0) {
      const uint32_t id = idesc(KIND, 128, p.NT, 0, 0);
      int stage = 0;
      uint32_t fphase = 0;
      int acc = 0;
      uint32_t aphase = 0;
      bool ok = true;
      bool issued_any = false;
      for (long long t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
        const TileCoord tc = decode_tile(p, t);
        const int ntaps = p.ph_ntaps[tc.ph];
        if (ntaps == 0) continue;
        const int tap0 = p.ph_tap_begin[tc.ph];
        if (!mbar_wait(bar_at(sm.acce, acc), aphase ^ 1u, abort_flag, &g_tap_err)) break;
        tc_fence_after();
        const uint32_t dcol = tmem + (uint32_t)(acc * p.MH * p.NT);
        for (int kb = 0; kb < p.nkb; ++kb) {
          if (!mbar_wait(bar_at(sm.full, stage), fphase, abort_flag, &g_tap_err) ||
              !mbar_wait(bar_at(sm.bfull, stage), fphase, abort_flag, &g_tap_err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          fence_proxy_async();
          const uint32_t a_st = sm.a0 + (uint32_t)stage * p.a_stage_bytes;
          const uint32_t b_st = sm.b0 + (uint32_t)stage * p.b_stage_bytes;
          if (NCH >= 2) {
            for (int ti = 0; ti < ntaps; ++ti) {
              const int tap = tap0 + ti;
              const uint32_t a_pl = a_st + (uint32_t)(p.tap_plane[tap] * NCH * rows) * 16u +
                                    (uint32_t)p.tap_off[tap] * 16u;
              const uint32_t b_tp = b_st + (uint32_t)(ti * b_tap_bytes);
              for (int ks = 0; ks < NCH / 2; ++ks) {
                const uint64_t bd =
                    sdesc(b_tp + (uint32_t)(2 * ks * p.NT) * 16u, (uint32_t)p.NT * 16u, 128u);
                const uint32_t first = (kb == 0 && ti == 0 && ks == 0) ? 0u : 1u;
                for (int h = 0; h < p.MH; ++h) {
                  const uint64_t ad = sdesc(a_pl + (uint32_t)(2 * ks * rows) * 16u + (uint32_t)(h * 128) * 16u,
                                            (uint32_t)rows * 16u, 128u);
                  mma_ss<KIND>(dcol + (uint32_t)(h * p.NT), ad, bd, id, first);
                }
              }
            }
          } else {
            // One channel chunk per tap: one MMA K-step covers two taps.  Its second
            // K-chunk is the next tap's rows, reached through the descriptor's chunk
            // stride (taps are sorted by staged address; a padding tap with zero
            // weights repeats the last address).
            for (int ti = 0; ti < ntaps; ti += 2) {
              const int t0 = tap0 + ti, t1 = t0 + 1;
              const uint32_t a0 = a_st + (uint32_t)(p.tap_plane[t0] * rows + p.tap_off[t0]) * 16u;
              const uint32_t a1 = a_st + (uint32_t)(p.tap_plane[t1] * rows + p.tap_off[t1]) * 16u;
              const uint64_t bd = sdesc(b_st + (uint32_t)(ti * b_tap_bytes), (uint32_t)p.NT * 16u, 128u);
              const uint32_t first = (kb == 0 && ti == 0) ? 0u : 1u;
              for (int h = 0; h < p.MH; ++h) {
                const uint64_t ad = sdesc(a0 + (uint32_t)(h * 128) * 16u, a1 - a0, 128u);
                mma_ss<KIND>(dcol + (uint32_t)(h * p.NT), ad, bd, id, first);
              }
            }
          }
          tc_commit(bar_at(sm.empty, stage));
          issued_any = true;
          if (++stage == S) {
            stage = 0;
            fphase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(bar_at(sm.accf, acc));
        if (++acc == p.ACCB) {
          acc = 0;
          aphase ^= 1u;
        }
      }
      if (!ok && issued_any) {
        // Wait (bounded) for every MMA already issued before TMEM is released.
        tc_commit(sm.drain);
        mbar_wait_drain(sm.drain, 0);
      }
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
  }
}

// ---------------------------------------------------------------------------- packing
// wpack chunk index = (((nt * nkb + kb) * ntaps + t) * NCH + j) * NT + n; the chunk holds
// CHUNK consecutive source channels cs = kb*CB + j*CHUNK + e of out channel nt*NT + n
// for filter tap (tap_r[t], tap_s[t]); zero outside the tensor.  fp32 values are
// rounded to tf32 (round to nearest, ties away) on the way.
template <int DT>
__global__ void pack_filter_kernel(const __grid_constant__ PackPlan pp) {
  constexpr int ESZ = DT == 0 ? 4 : 2;
  constexpr int CHUNK = 16 / ESZ;
  const int NCH = pp.CB / CHUNK;
  const long long total = (long long)pp.n_ntiles * pp.nkb * pp.ntaps_total * NCH * pp.NT;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    long long rest = idx;
    const int n = (int)(rest % pp.NT);
    rest /= pp.NT;
    const int j = (int)(rest % NCH);
    rest /= NCH;
    const int t = (int)(rest % pp.ntaps_total);
    rest /= pp.ntaps_total;
    const int kb = (int)(rest % pp.nkb);
    const int nt = (int)(rest / pp.nkb);
    const int nn = nt * pp.NT + n;
    const int r = pp.tap_r[t], s = pp.tap_s[t];
    uint32_t out[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int e = 0; e < CHUNK; ++e) {
      const int cs = kb * pp.CB + j * CHUNK + e;
      if (nn < pp.Cd && cs < pp.Cs && r >= 0) {
        const long long widx = pp.transpose ? (((long long)cs * pp.C + nn) * pp.R + r) * pp.S + s
                                            : (((long long)nn * pp.C + cs) * pp.R + r) * pp.S + s;
        if constexpr (DT == 0) {
          const float v = static_cast<const float*>(pp.w)[widx];
          uint32_t tf;
          asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(tf) : "f"(v));
          out[e] = tf;
        } else {
          const uint32_t v = static_cast<const uint16_t*>(pp.w)[widx];
          out[e >> 1] |= v << (16 * (e & 1));
        }
      }
    }
    reinterpret_cast<uint4*>(pp.wpack)[idx] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// ---------------------------------------------------------------------------- launchers
size_t tap_gemm_smem_bytes(const TapPlan& p) {
  size_t b = (size_t)p.stages * (p.a_stage_bytes + p.b_stage_bytes);
  b += (size_t)p.npl * p.rows * sizeof(int);
  b = (b + 15) & ~size_t(15);
  b += 8 * (3 * p.stages + 5) + 16;
  return b + 1024;  // alignment slack for the dynamic base
}

cudaError_t launch_tap_gemm(const TapPlan& p, int dt, int grid, cudaStream_t st) {
  const size_t smem = tap_gemm_smem_bytes(p);
  cudaError_t e;
  if (dt == 0) {
    e = cudaFuncSetAttribute(tap_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    tap_gemm_kernel<0><<<grid, kThreads, smem, st>>>(p);
  } else {
    e = cudaFuncSetAttribute(tap_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    tap_gemm_kernel<1><<<grid, kThreads, smem, st>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_pack_filter(const PackPlan& pp, int dt, cudaStream_t st) {
  const int CHUNK = dt == 0 ? 4 : 8;
  const long long total = (long long)pp.n_ntiles * pp.nkb * pp.ntaps_total * (pp.CB / CHUNK) * pp.NT;
  long long blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  if (dt == 0)
    pack_filter_kernel<0><<<(int)blocks, 256, 0, st>>>(pp);
  else
    pack_filter_kernel<1><<<(int)blocks, 256, 0, st>>>(pp);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------- fixed scratch
// Filter-pack scratch for conv2d_fwd_noalloc: a file-scope device array, so that callers
// who cannot allocate device memory can still run the forward op.  Every GPU that loads
// this library holds it until the process exits.  Host code must not pass the array's
// name to a kernel (on the host it is only a stand-in); the device address is looked up
// once per device with cudaGetSymbolAddress while that device is current.
constexpr size_t kNoAllocScratchBytes = 8u << 20;  // 8 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

size_t noalloc_scratch_capacity() { return kNoAllocScratchBytes; }

// Device address of the scratch on the current device (looked up on first use per
// device, then cached).  Returns cudaSuccess and sets *ptr, or the lookup's error.
cudaError_t noalloc_scratch_ptr(void** ptr) {
  static std::mutex mu;
  static std::vector<void*> cache;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  if ((size_t)dev < cache.size() && cache[dev] != nullptr) {
    *ptr = cache[dev];
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  if ((size_t)dev >= cache.size()) cache.resize(dev + 1, nullptr);
  cache[dev] = p;
  *ptr = p;
  return cudaSuccess;
}

int tap_gemm_take_error() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_tap_err, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) cudaMemcpyToSymbol(g_tap_err, &zero, sizeof(int));
  return v;
}

}  // namespace cg3

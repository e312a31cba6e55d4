// conv_wgrad_mn.cu -- backward-filter of bf16 tensors on channel-chunked planes (sm_103a).
//
//   dw[k,c,r,s] = sum_{n,p,q} X(n, c, p*sh - ph + r*dh, q*sw - pw + s*dw) * dy[n,k,p,q]
// (the filter gradient of the cuDNN backward-filter call in Apache SystemDS
// LibMatrixCuDNNConvolutionAlgorithm.java; deconvolution's backward-weights in Apache MXNet
// mkldnn_deconvolution.cc is the same product with the weight's roles swapped).
//
// Two kernels:
//   nhwc_pack_kernel   copies an NCHW tensor into zero-padded planes whose 16-byte groups hold
//                      consecutive channels of one position (see NhwcPackPlan); x goes in once
//                      per stride phase plane, dy once.
//   wgrad_mn_kernel    one implicit GEMM per tile over the padded position space (WgradMnPlan):
//                      a single thread stages, per pipeline stage, one x tile (128 channels x
//                      the stage's positions plus the tap group's span) and one dy tile (NK
//                      output channels x the stage's positions) with tensor copies; both land
//                      in the MN-major operand layout (16 bytes = 8 channels of one position,
//                      8 positions per core matrix), so every tap of the group is the same x
//                      tile started a few rows later.  One elected thread issues, per 16
//                      positions and tap, one tcgen05.mma kind::f16 (bf16 operands, fp32
//                      accumulators in TMEM, M = 128 channels, N = NK); four epilogue warps
//                      move each tap's accumulator to the fp32 split partials, which the
//                      fixed-order reduce of conv_wgrad.cu adds into dw.
#include <algorithm>
#include <atomic>
#include <type_traits>

#include <cuda_bf16.h>

#include "conv_pack.cuh"
#include "conv_plan.h"
#include "sm103_ptx.cuh"
#include "launch_util.cuh"

namespace cg3 {

__device__ int g_wgmn_err;

namespace {

constexpr int kMnEpiWarps = 8;    // two per TMEM lane quarter, taking alternate 16-column chunks
constexpr int kMnThreads = 32 * (2 + kMnEpiWarps);  // warp 0 producer, warp 1 TMEM + MMA, then epilogue
constexpr int kMnRowPitch = 80;   // epilogue staging: 16 fp32 + 16 bytes per row (conflict-free)
constexpr int kMnStageTile = 32 * kMnRowPitch;

__device__ __forceinline__ uint32_t bar_at(uint32_t base, int i) { return base + 8u * (uint32_t)i; }

struct MnTile {
  int sp, g, mc, nk;
};

// Tiles run output-channel tile fastest, then channel tile, tap group and split, so that CTAs
// running at the same time share their x tiles (same channel tile) and dy tiles (same split).
__device__ __forceinline__ MnTile decode_mn(const WgradMnPlan& p, long long t) {
  MnTile w;
  w.nk = (int)(t % p.n_ktiles);
  long long r = t / p.n_ktiles;
  w.mc = (int)(r % p.n_ctiles);
  r /= p.n_ctiles;
  w.g = (int)(r % p.ngroups);
  w.sp = (int)(r / p.ngroups);
  return w;
}

// One stage's MMAs: for every tap j of the group, KS steps of 16 positions (unrolled; a single
// issuing thread spends tens of cycles per tcgen05.mma in a runtime-bounded loop).
template <int KS>
__device__ __forceinline__ void issue_mn_stage(const WgradMnPlan& p, uint32_t tmem, uint32_t xlo, uint32_t ylo,
                                               uint32_t a_hi, uint32_t b_hi, uint32_t id, int tap0, int ntaps,
                                               bool first) {
  for (int j = 0; j < ntaps; ++j) {
    const uint32_t d = tmem + (uint32_t)(j * p.NK);
    const uint32_t alo = xlo + (uint32_t)p.tap_delta[tap0 + j];  // 16-byte units
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
      mma_ss_lh<1>(d, alo + 16u * ks, a_hi, ylo + 16u * ks, b_hi, id, (first && ks == 0) ? 0u : 1u);
  }
}

}  // namespace

// Channel-chunk packs of plan `a` and (b.src not NULL) plan `b` in one launch: the units of `a`,
// then those of `b`, one per block iteration (nhwc_pack_unit).
template <int DT>
__global__ void __launch_bounds__(256) nhwc_pack_kernel(const __grid_constant__ NhwcPackPlan a,
                                                        const __grid_constant__ NhwcPackPlan b) {
  extern __shared__ __align__(16) uint8_t pk_smem[];
  const uint32_t na = a.units, nb = b.src != nullptr ? b.units : 0u;
  for (uint32_t u = blockIdx.x; u < na + nb; u += gridDim.x) {
    if (u < na)
      nhwc_pack_unit<DT>(a, u, pk_smem);
    else
      nhwc_pack_unit<DT>(b, u - na, pk_smem);
  }
}

// Fixed-order sum of the split partials and transpose into KCRS (ReduceTPlan): a block of 8 warps
// takes a tile of 32 partial rows (c, tap) x 128 output channels k; lane l of warp w adds, in
// split order, the 4 consecutive k (one 16-byte read per split: a warp reads 512 contiguous
// bytes of a row) of rows w, w + 8, w + 16, w + 24; the tile is transposed through shared memory
// and each warp writes runs of 32 consecutive dw elements (rows) per k.  K % 4 == 0.
template <int DT, bool GRP>  // GRP: rp.gk != 0 (grouped: diagonal blocks only)
__global__ void __launch_bounds__(256) wgrad_reduce_t_kernel(const __grid_constant__ ReduceTPlan rp) {
  __shared__ float tile[32][129];
  griddep_wait();  // the partials are written by the previous grid
  const int tx = (int)(threadIdx.x & 31), ty = (int)(threadIdx.x >> 5);
  const long long ntr = (rp.rows + 31) / 32, ntk = (rp.K + 127) / 128;
  const long long split_stride = (long long)rp.rows * rp.K;
  for (long long tid = blockIdx.x; tid < ntr * ntk; tid += gridDim.x) {
    const int r0 = (int)(tid / ntk) * 32, k0 = (int)(tid % ntk) * 128;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    const int k = k0 + 4 * tx;
    if (k < rp.K) {
      const float* src = rp.partial + k;
      for (int sp = 0; sp < rp.nsplit; ++sp) {
        float4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = r0 + ty + 8 * i;
          v[i] = row < rp.rows ? __ldg(reinterpret_cast<const float4*>(src + (long long)sp * split_stride +
                                                                        (long long)row * rp.K))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[i][0] += v[i].x;
          acc[i][1] += v[i].y;
          acc[i][2] += v[i].z;
          acc[i][3] += v[i].w;
        }
      }
    }
    __syncthreads();  // the previous tile's transposed values are read
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) tile[ty + 8 * i][4 * tx + j] = acc[i][j];
    __syncthreads();
    for (int kk = ty; kk < 128; kk += 8) {
      const int kg = k0 + kk, row = r0 + tx;
      if (kg >= rp.K || row >= rp.rows) continue;
      float v = tile[tx][kk];
      int orow = row;
      if (rp.flip) {
        const int c = row / rp.RS;
        orow = c * rp.RS + (rp.RS - 1 - (row - c * rp.RS));
      }
      long long o = (long long)kg * rp.rows + orow;
      if constexpr (GRP) {  // grouped: keep the diagonal block of k's group
        const int g = kg / rp.gk;
        if (row / rp.RS / rp.gc != g) continue;
        o = ((long long)kg * rp.gc - (long long)g * rp.gc) * rp.RS + orow;
      }
      if constexpr (DT == 0) {
        float* dwp = static_cast<float*>(rp.dw);
        if (rp.beta != 0.f) v += rp.beta * dwp[o];
        dwp[o] = v;
      } else {
        __nv_bfloat16* dwp = static_cast<__nv_bfloat16*>(rp.dw);
        if (rp.beta != 0.f) v += rp.beta * __bfloat162float(dwp[o]);
        dwp[o] = __float2bfloat16_rn(v);
      }
    }
  }
}

__global__ void __launch_bounds__(kMnThreads, 1) wgrad_mn_kernel(const __grid_constant__ WgradMnPlan p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int S = p.stages;
  const int KB = p.KB;

  uint8_t* ptr = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t a0 = smem_u32(ptr);  // x tiles, one per stage (1024-byte multiples)
  ptr += (size_t)S * p.a_stage_bytes;
  const uint32_t b0 = smem_u32(ptr);  // dy tiles
  ptr += (size_t)S * p.b_stage_bytes;
  const uint32_t stg0 = smem_u32(ptr);  // epilogue: one 32 x 32 fp32 tile per warp, rows 144 bytes apart
  ptr += kMnStageTile * kMnEpiWarps;
  const uint32_t full = smem_u32(ptr);
  const uint32_t empty = full + 8u * S;
  const uint32_t accf = empty + 8u * S;
  const uint32_t acce = accf + 8u;
  const uint32_t drain = acce + 8u;
  ptr += 8 * (2 * S + 3);
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(ptr);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ptr + 4);
  // The carve-up must lie inside the launch's dynamic shared memory; otherwise record the error
  // and leave before touching any of it (every thread takes the same branch).
  if ((uint32_t)(ptr + 8 - smem_raw) > dynamic_smem_bytes()) {
    if (tid == 0) atomicExch(&g_wgmn_err, DEV_ERR_LAYOUT);
    return;
  }

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_at(full, s), 1);   // the producer's arrival + both copies' bytes
      mbar_init(bar_at(empty, s), 1);  // the MMA commit
    }
    mbar_init(accf, 1);
    mbar_init(acce, kMnEpiWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32((const void*)tmem_holder), (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  griddep_launch_dependents();  // the reduce may be scheduled; it waits for this grid to finish

  if (warp == 0) {
    // =============================================================== producer (one thread)
    if (lane == 0) {
      uint32_t last[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};  // 1 + parity of the last fill per slot
      const uint32_t bytes = (uint32_t)p.tx_bytes;  // both boxes, out-of-bounds parts included
      long long counter = 0;
      bool ok = true;
      for (long long t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
        const MnTile w = decode_mn(p, t);
        const long long lbeg = (long long)w.sp * p.split_len;
        const long long lend = lbeg + p.split_len < p.Mtot ? lbeg + p.split_len : p.Mtot;
        const int xoff = p.grp_off0[w.g];
        for (long long l0 = lbeg; l0 < lend; l0 += KB, ++counter) {
          const int stage = (int)(counter % S);
          const uint32_t ephase = (uint32_t)((counter / S) & 1);
          if (!mbar_wait(bar_at(empty, stage), ephase ^ 1u, abort_flag, &g_wgmn_err)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_at(full, stage);
          mbar_arrive_expect_tx(fb, bytes);
          // boxes past the position space or the channel extents read as zeros
          tma_load_3d(a0 + (uint32_t)stage * (uint32_t)p.a_stage_bytes, &p.tm_x, (int)(2 * (l0 + xoff)), 16 * w.mc,
                      p.grp_plane[w.g], fb);
          tma_load_2d(b0 + (uint32_t)stage * (uint32_t)p.b_stage_bytes, &p.tm_dy, (int)(2 * l0), (p.NK / 8) * w.nk, fb);
          if (stage < 8) last[stage] = 1u + ephase;
        }
      }
      // After an abort, wait (bounded) for copies still in flight into shared memory.
      if (*abort_flag)
        for (int s = 0; s < S && s < 8; ++s)
          if (last[s]) mbar_wait_drain(bar_at(full, s), last[s] - 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // =============================================================== MMA issuer
    const bool leader = elect_one();
    const uint32_t id = idesc(1, 128, p.NK, 1, 1);  // bf16 x bf16 -> fp32, both operands MN-major
    const uint32_t a_hi = (uint32_t)(sdesc(0u, 0u, (uint32_t)(p.KBX * 16)) >> 32);  // stride offset + version
    const uint32_t b_hi = (uint32_t)(sdesc(0u, 0u, (uint32_t)(KB * 16)) >> 32);
    long long counter = 0;
    uint32_t aphase = 0;
    bool ok = true, issued = false;
    for (long long t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
      const MnTile w = decode_mn(p, t);
      const long long lbeg = (long long)w.sp * p.split_len;
      const long long lend = lbeg + p.split_len < p.Mtot ? lbeg + p.split_len : p.Mtot;
      const int tap0 = p.grp_tap0[w.g], ntaps = p.grp_ntaps[w.g];
      // the epilogue has moved the previous tile's accumulators out of TMEM
      if (!mbar_wait(acce, aphase ^ 1u, abort_flag, &g_wgmn_err)) break;
      tc_fence_after();
      bool first = true;
      for (long long l0 = lbeg; l0 < lend; l0 += KB, ++counter) {
        const int stage = (int)(counter % S);
        const uint32_t fphase = (uint32_t)((counter / S) & 1);
        if (!mbar_wait(bar_at(full, stage), fphase, abort_flag, &g_wgmn_err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (leader) {
          // descriptor low halves (start address, leading offset 128 B) of the stage's tiles; a
          // tap starts its x tile tap_delta rows later, a 16-position step is 16 rows
          const uint32_t xlo = (uint32_t)sdesc(a0 + (uint32_t)stage * (uint32_t)p.a_stage_bytes, 128u, 0u);
          const uint32_t ylo = (uint32_t)sdesc(b0 + (uint32_t)stage * (uint32_t)p.b_stage_bytes, 128u, 0u);
          switch (KB / 16) {
            case 2: issue_mn_stage<2>(p, tmem, xlo, ylo, a_hi, b_hi, id, tap0, ntaps, first); break;
            case 4: issue_mn_stage<4>(p, tmem, xlo, ylo, a_hi, b_hi, id, tap0, ntaps, first); break;
            default: issue_mn_stage<8>(p, tmem, xlo, ylo, a_hi, b_hi, id, tap0, ntaps, first); break;
          }
          tc_commit(bar_at(empty, stage));  // frees the stage once its MMAs are done
        }
        __syncwarp();
        issued = true;
        first = false;
      }
      if (!ok) break;
      if (leader) tc_commit(accf);
      __syncwarp();
      aphase ^= 1u;
    }
    if (!ok && issued && leader) {
      tc_commit(drain);
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  } else {
    // =============================================================== epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const bool vec = (p.K & 3) == 0;
    uint32_t aphase = 0;
    for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
      const MnTile w = decode_mn(p, t);
      if (!mbar_wait(accf, aphase, abort_flag, &g_wgmn_err)) break;
      tc_fence_after();
      // Each warp moves its 32 TMEM lanes (channels c) 16 columns at a time (the two warps of a
      // lane quarter take alternate chunks): TMEM -> registers -> a padded shared tile (lane = row)
      // -> registers (4 lanes per row) -> 64 contiguous bytes of each of 8 partial rows per store
      // instruction.  The next chunk's TMEM load is in flight while a chunk is stored.
      const int c_w = 128 * w.mc + 32 * q;  // first channel of this warp's rows
      const int tap0 = p.grp_tap0[w.g], ntaps = p.grp_ntaps[w.g];
      const uint32_t stg = stg0 + (uint32_t)((warp - 2) * kMnStageTile);
      const int half = (warp - 2) >> 2;
      const int rr = lane >> 2, ch = lane & 3;  // read-back: row within a group of 8, 16-byte chunk
      const int nchunk = p.NK / 16;             // per tap
      const int total = ntaps * nchunk;
      uint32_t ra[16], rb[16];
      int ci = half;
      if (ci < total)
        tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)((ci / nchunk) * p.NK + 16 * (ci % nchunk)), ra);
      while (ci < total) {
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) rb[i] = ra[i];
        const int nx = ci + 2;
        if (nx < total)
          tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)((nx / nchunk) * p.NK + 16 * (nx % nchunk)), ra);
        const int j = ci / nchunk, c0 = 16 * (ci % nchunk);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(stg + (uint32_t)(lane * kMnRowPitch + 16 * i)),
                       "r"(rb[4 * i]), "r"(rb[4 * i + 1]), "r"(rb[4 * i + 2]), "r"(rb[4 * i + 3])
                       : "memory");
        __syncwarp();
        const long long row0 = ((long long)w.sp * p.C + c_w) * p.RS + p.tap_out[tap0 + j];  // partial row of c_w
        const int kk = w.nk * p.NK + c0 + 4 * ch;  // this lane's 4 output channels
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int row = 8 * g + rr;  // channel c_w + row
          uint32_t v0, v1, v2, v3;
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                       : "r"(stg + (uint32_t)(row * kMnRowPitch + 16 * ch)));
          if (c_w + row < p.C && kk < p.K) {
            float* d = p.partial + (row0 + (long long)row * p.RS) * p.K + kk;
            if (vec) {
              *reinterpret_cast<uint4*>(d) = make_uint4(v0, v1, v2, v3);
            } else {
              const uint32_t vv[4] = {v0, v1, v2, v3};
#pragma unroll
              for (int i = 0; i < 4; ++i)
                if (kk + i < p.K) d[i] = __uint_as_float(vv[i]);
            }
          }
        }
        __syncwarp();
        ci = nx;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce);
      aphase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
  }
}

// ---------------------------------------------------------------------------- launchers
// A CTA that takes more than half of TMEM asks for more than half of the SM's shared memory,
// so that a second CTA never waits on the SM for TMEM columns.
size_t wgrad_mn_smem_bytes(const WgradMnPlan& p) {
  const size_t b = (size_t)p.stages * (p.a_stage_bytes + p.b_stage_bytes) + (size_t)kMnEpiWarps * kMnStageTile +
                   8 * (2 * p.stages + 3) + 16 + 1024;
  return p.tmem_cols > 256 && b < (size_t)(120 << 10) ? (size_t)(120 << 10) : b;
}

static std::atomic<int> g_mn_smem_set[kMaxDevices];

cudaError_t launch_wgrad_mn(const WgradMnPlan& p, int grid, cudaStream_t st) {
  const size_t smem = wgrad_mn_smem_bytes(p);
  const cudaError_t e = ensure_dyn_smem(wgrad_mn_kernel, smem, g_mn_smem_set);
  if (e != cudaSuccess) return e;
  wgrad_mn_kernel<<<grid, kMnThreads, smem, st>>>(p);
  return cudaGetLastError();
}

// Packs a and (if b.src is not NULL) b in one launch.
cudaError_t launch_nhwc_pack(const NhwcPackPlan& a, const NhwcPackPlan& b, int dt, int num_sms, cudaStream_t st) {
  const bool two = b.src != nullptr;
  const size_t smem = std::max(nhwc_pack_smem_bytes(a, dt), two ? nhwc_pack_smem_bytes(b, dt) : (size_t)0);
  const long long units = (long long)a.units + (two ? (long long)b.units : 0ll);
  const long long per_sm = std::max<long long>(1, std::min<long long>(8, (long long)(200 * 1024) / (long long)std::max<size_t>(smem, 1)));
  const unsigned blocks = (unsigned)std::max(1ll, std::min<long long>(units, (long long)num_sms * per_sm));
  static std::atomic<int> set_bytes[2][kMaxDevices];
  cudaError_t e;
  if (dt == 0) {
    e = ensure_dyn_smem(nhwc_pack_kernel<0>, smem, set_bytes[0]);
    if (e != cudaSuccess) return e;
    nhwc_pack_kernel<0><<<blocks, 256, smem, st>>>(a, b);
  } else {
    e = ensure_dyn_smem(nhwc_pack_kernel<1>, smem, set_bytes[1]);
    if (e != cudaSuccess) return e;
    nhwc_pack_kernel<1><<<blocks, 256, smem, st>>>(a, b);
  }
  return cudaGetLastError();
}

// Launched with programmatic stream serialization after the GEMM (it waits for the GEMM).
cudaError_t launch_wgrad_reduce_t(const ReduceTPlan& rp, int dt, int num_sms, cudaStream_t st) {
  const long long tiles = (long long)(rp.rows + 31) / 32 * ((rp.K + 127) / 128);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::max(1ll, std::min<long long>(tiles, (long long)num_sms * 8)));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool grp = rp.gk != 0;
  const cudaError_t e = dt == 0 ? (grp ? cudaLaunchKernelEx(&cfg, wgrad_reduce_t_kernel<0, true>, rp)
                                       : cudaLaunchKernelEx(&cfg, wgrad_reduce_t_kernel<0, false>, rp))
                                : (grp ? cudaLaunchKernelEx(&cfg, wgrad_reduce_t_kernel<1, true>, rp)
                                       : cudaLaunchKernelEx(&cfg, wgrad_reduce_t_kernel<1, false>, rp));
  return e != cudaSuccess ? e : cudaGetLastError();
}

int wgrad_mn_take_error() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_wgmn_err, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) cudaMemcpyToSymbol(g_wgmn_err, &zero, sizeof(int));
  return v;
}

}  // namespace cg3

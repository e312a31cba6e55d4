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
// CTA roles (448 threads, persistent over tiles):
//   warps 0-7  two producer groups taking pipeline stages in turn: stage source rows
//              for CB channels into shared memory in the core-matrix interleaved layout,
//              and bulk-copy the packed filter slice.  The rows come either from a copy of
//              the source packed channel-chunk-wise beforehand (nhwc pack kernel), by
//              tensor copies of whole runs of rows, or straight from NCHW (one load per
//              channel of each staged row, 16-byte shared stores) when the caller gives
//              no room for that copy.
//   warps 8-11 epilogue: TMEM -> registers -> NCHW global stores, coalesced along
//              output positions, with the optional bias and add-to (beta) of the fused
//              epilogue; bf16 outputs rounded to nearest even.
//   warps 12-13 TMEM allocation (warp 12); each warp issues tcgen05.mma (kind::tf32
//              for fp32, kind::f16 with bf16 operands) for one 128-row accumulator half,
//              through one elected lane.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "conv_pack.cuh"
#include "conv_plan.h"
#include "conv_stage.cuh"
#include "sm103_ptx.cuh"
#include "launch_util.cuh"

namespace cg3 {

__device__ int g_tap_err;

namespace {

// CTA roles: warps 0-7 two producer groups (group g fills the stages with global stage
// counter = g mod 2), warps 8-11 epilogue, warp 12 TMEM allocation + MMA issue for the
// first 128-row half of a tile, warp 13 MMA issue for the second half.
constexpr int kThreads = 448;
constexpr int kProdThreads = 128;  // per producer group
constexpr int kEpiWarp0 = 8;
constexpr int kMmaWarp = 12;

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
__device__ __forceinline__ float load_elem(const void* base, long long idx) {
  if constexpr (DT == 0)
    return static_cast<const float*>(base)[idx];
  else
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[idx]);
}

// Fused epilogue of 16 output channels (the first `lim` of them exist) at one output position,
// with the old values and the channels' bias values (zero without bias) already read:
// D + bias (+ beta * old), in fp32, then stored (bf16: rounded to nearest even).
template <int DT>
__device__ __forceinline__ void store16_epi(const TapPlan& p, long long ob, long long ostep, int lim,
                                            const uint32_t (&r)[16], const float (&old)[16], const float (&bv)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j < lim) {
      float v = __uint_as_float(r[j]) + bv[j];
      if (p.beta != 0.f) v += p.beta * old[j];
      if constexpr (DT == 0)
        static_cast<float*>(p.dst)[ob + j * ostep] = v;
      else
        static_cast<__nv_bfloat16*>(p.dst)[ob + j * ostep] = __float2bfloat16_rn(v);
    }
  }
}

// Epilogue of 16 output channels ch0 .. ch0 + 15 (the first `lim` of them exist) at one output
// position: D (+ bias of the channel) (+ beta * the old value), in fp32, then stored (bf16:
// rounded to nearest even).  The old values are all read before the first store, so their
// reads overlap instead of each waiting behind the previous store.
template <int DT, bool EPI>
__device__ __forceinline__ void store16(const TapPlan& p, long long ob, long long ostep, int ch0, int lim,
                                        const uint32_t (&r)[16]) {
  if constexpr (!EPI) {
    auto st1 = [&](int j) {
      if constexpr (DT == 0)
        static_cast<float*>(p.dst)[ob + j * ostep] = __uint_as_float(r[j]);
      else
        static_cast<__nv_bfloat16*>(p.dst)[ob + j * ostep] = __float2bfloat16_rn(__uint_as_float(r[j]));
    };
    if (lim >= 16) {
#pragma unroll
      for (int j = 0; j < 16; ++j) st1(j);
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < lim) st1(j);
    }
    return;
  }
  float old[16];
  if (p.beta != 0.f) {
#pragma unroll
    for (int j = 0; j < 16; ++j) old[j] = j < lim ? load_elem<DT>(p.dst, ob + j * ostep) : 0.f;
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j < lim) {
      float v = __uint_as_float(r[j]);
      if (p.bias != nullptr) v += load_elem<DT>(p.bias, ch0 + j);
      if (p.beta != 0.f) v += p.beta * old[j];
      if constexpr (DT == 0)
        static_cast<float*>(p.dst)[ob + j * ostep] = v;
      else
        static_cast<__nv_bfloat16*>(p.dst)[ob + j * ostep] = __float2bfloat16_rn(v);
    }
  }
}

// Issues one pipeline stage's MMAs for one 128-row accumulator, by the elected lane alone: for
// every tap of the phase (four at a time, straight-line), KS MMAs (K = two 16-byte chunks each)
// over the stage's channel chunks; KS == 0 is tap-pair mode (one MMA covers two taps whose rows
// the A entry's chunk stride links).  The taps' operand offsets are read from the kernel
// parameters: a constant-cache read, which does not wait behind the MMAs this thread has issued
// (a shared-memory load would).  A single issuing thread spends tens of cycles per tcgen05.mma,
// more in a loop with shuffles or branches, so the sequence is kept short and unrolled.
template <int KIND, int KS>
__device__ __forceinline__ void issue_stage(const TapPlan& p, int tap0, int ntaps, uint32_t dcol, uint32_t a_lo0,
                                            uint32_t b_lo0, uint32_t d_hi, uint32_t id, uint32_t a_ks, uint32_t b_ks,
                                            bool first) {
  constexpr int TSTEP = KS == 0 ? 2 : 1;
  auto one = [&](int t, bool init) {
    const uint32_t alo = a_lo0 + (uint32_t)p.tap_a[t], blo = b_lo0 + (uint32_t)p.tap_b[t];
    if constexpr (KS == 0) {
      mma_ss_lh<KIND>(dcol, alo, d_hi, blo, d_hi, id, init ? 0u : 1u);
    } else {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
        mma_ss_lh<KIND>(dcol, alo + (uint32_t)ks * a_ks, d_hi, blo + (uint32_t)ks * b_ks, d_hi, id,
                        (init && ks == 0) ? 0u : 1u);
    }
  };
  int j = 0;
  for (; j + 4 * TSTEP <= ntaps; j += 4 * TSTEP) {
#pragma unroll
    for (int u = 0; u < 4; ++u) one(tap0 + j + u * TSTEP, first && j == 0 && u == 0);
  }
  for (; j < ntaps; j += TSTEP) one(tap0 + j, first && j == 0);
}

}  // namespace

// EPI: the launch has a bias or beta != 0 (fused epilogue); the plain kernel stores D only.
template <int DT, bool EPI>
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
  const uint32_t a0 = smem_u32(ptr);
  ptr += (size_t)S * p.a_stage_bytes;
  const uint32_t b0 = smem_u32(ptr);
  ptr += (size_t)S * p.b_stage_bytes;
  ptr = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ptr) + 15) & ~uintptr_t(15));
  const uint32_t full = smem_u32(ptr);
  const uint32_t empty = full + 8u * S;
  const uint32_t accf = empty + 8u * S;
  const uint32_t acce = accf + 16u;
  const uint32_t drain = acce + 16u;  // two entries, one per issuer
  ptr += 8 * (2 * S + 6);
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(ptr);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ptr + 4);
  // Per stage slot: 0 = never used, else 1 + parity of the last bulk copy issued into it.
  volatile int* last_copy = reinterpret_cast<volatile int*>(ptr + 8);

  const int nissuers = p.MH;  // one MMA-issuing thread per 128-row accumulator half
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_at(full, s), kProdThreads);  // + the filter copy's transaction bytes
      mbar_init(bar_at(empty, s), (uint32_t)nissuers);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_at(accf, a), (uint32_t)nissuers);
      mbar_init(bar_at(acce, a), 4);
    }
    mbar_init(drain, 1);
    mbar_init(drain + 8u, 1);
    *abort_flag = 0;
    for (int s = 0; s < S; ++s) last_copy[s] = 0;
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

  const long long HdWd = (long long)p.Hd * p.Wd;
  const int MT = 128 * p.MH;
  const int b_tap_bytes = NCH * p.NT * 16;

  if (warp < kEpiWarp0) {
    // =============================================================== producers
    const int grp = warp >> 2;           // producer group 0 or 1
    const int gtid = tid & (kProdThreads - 1);
    if (gtid == 0) griddep_wait();       // the packed filter is written by the previous grid
    long long counter = 0;               // global stage counter (both groups count all stages)
    bool ok = true;
    // After an abort a group keeps walking the tiles (skipping all work) to the final
    // named barrier below instead of leaving early.
    for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
      const TileCoord tc = decode_tile(p, t);
      const int ntaps = p.ph_ntaps[tc.ph];
      if (ntaps == 0) continue;
      const long long m0 = (long long)tc.mt * MT;
      for (int kb = 0; kb < p.nkb; ++kb, ++counter) {
        if ((int)(counter & 1) != grp || !ok) continue;
        const int stage = (int)(counter % S);
        const uint32_t ephase = (uint32_t)((counter / S) & 1);
        if (!mbar_wait(bar_at(empty, stage), ephase ^ 1u, abort_flag, &g_tap_err)) {
          ok = false;
          continue;
        }
        const uint32_t a_st = a0 + (uint32_t)stage * p.a_stage_bytes;
        const uint32_t b_st = b0 + (uint32_t)stage * p.b_stage_bytes;
        if (gtid == 0) {
          const uint32_t bytes = (uint32_t)(ntaps * b_tap_bytes);
          const long long img_off =
              ((long long)(tc.nt * p.nkb + kb) * p.ntaps_total + p.ph_tap_begin[tc.ph]) * b_tap_bytes;
          // The copies complete on the stage's full barrier: their bytes are expected there
          // before they are issued, and this thread arrives with the others after its fill.
          mbar_expect_tx(bar_at(full, stage), bytes + (p.a_tma ? (uint32_t)p.a_stage_bytes : 0u));
          bulk_g2s(b_st, static_cast<const uint8_t*>(p.wpack) + img_off, bytes, bar_at(full, stage));
          if (p.a_tma) {
            // one tensor copy per (plane, chunk, box of rows): [plane][chunk][row][16 bytes]; with a
            // shift per phase, the plane's rows from the tile's phase origin (a negative start
            // reads zeros)
            const long long l0 = m0 + (p.plane_per_phase ? p.ph_shift[tc.ph] : 0);
            if (p.a_one) {  // every plane and chunk of the stage in one copy, [plane][chunk][row]
              tma_load_4d(a_st, &p.tm_src, 0, (int)l0, kb * NCH, 0, bar_at(full, stage));
            } else {
              for (int pl = 0; pl < p.npl; ++pl)
                for (int j = 0; j < NCH; ++j)
                  for (int bx = 0; bx < p.a_nbox; ++bx)
                    tma_load_3d(a_st + (uint32_t)(((pl * NCH + j) * rows + bx * p.a_box) * 16), &p.tm_src,
                                (int)(2 * (l0 + (long long)bx * p.a_box)), kb * NCH + j, pl, bar_at(full, stage));
            }
          }
          last_copy[stage] = 1 + (int)ephase;
        }
        if (!p.a_tma) {
          stage_pixel_rows<DT>(p, m0, a_st, kb * p.CB, NCH, gtid);
          fence_proxy_async();
        }
        mbar_arrive(bar_at(full, stage));
      }
    }
    // After an abort, never leave a bulk copy in flight into shared memory that is about
    // to be released.  (In a normal run the MMA lane has waited on every copy.)  The copy
    // completes on the stage's full barrier together with the producers' arrivals, so
    // after an abort its phase may never complete: the bounded drain then gives up after
    // its time limit.  Slots are shared by both groups, so the last copy per slot is known
    // only after both groups are done issuing.
    named_bar_sync(1, 2 * kProdThreads);
    if (tid == 0 && *abort_flag) {
      for (int s = 0; s < S; ++s)
        if (last_copy[s]) mbar_wait_drain(bar_at(full, s), (uint32_t)(last_copy[s] - 1));
    }
  } else if (warp < kMmaWarp) {
    // =============================================================== epilogue
    const int q = warp & 3;
    int acc = 0;
    uint32_t aphase = 0;
    for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
      const TileCoord tc = decode_tile(p, t);
      const int ntaps = p.ph_ntaps[tc.ph];
      const long long m0 = (long long)tc.mt * MT;
      if constexpr (EPI) {
        // Add-to: while the tile's accumulator is computed, pull the old output values of
        // this lane's rows into L2 (the epilogue's reads of them then wait on L2, not DRAM).
        if (p.beta != 0.f) {
          const int nb = tc.nt * p.NT;
          const int nv = min(p.NT, p.Cd - nb);
          for (int h = 0; h < p.MH; ++h) {
            const long long L = m0 + h * 128 + q * 32 + lane;
            if (L >= p.Mtot) continue;
            const uint32_t n = fdiv((uint32_t)L, p.fd_img);
            const uint32_t rem = (uint32_t)L - n * p.fd_img.d;
            const int e = (int)fdiv(rem, p.fd_WL);
            const int f = (int)rem - e * p.WL;
            const int oh = e * p.ph_step_h + p.ph_off_h[tc.ph];
            const int ow = f * p.ph_step_w + p.ph_off_w[tc.ph];
            if (oh < 0 || oh >= p.Hd || ow < 0 || ow >= p.Wd) continue;
            const char* o = static_cast<const char*>(p.dst) +
                            ((long long)n * p.dst_nstride + (long long)nb * HdWd + (long long)oh * p.Wd + ow) * (DT == 0 ? 4 : 2);
            for (int j = 0; j < nv; ++j) prefetch_l2(o + (long long)j * HdWd * (DT == 0 ? 4 : 2));
          }
        }
      }
      if (ntaps != 0) {
        if (!mbar_wait(bar_at(accf, acc), aphase, abort_flag, &g_tap_err)) break;
        tc_fence_after();
      }
      for (int h = 0; h < p.MH; ++h) {
        const int m = h * 128 + q * 32 + lane;
        const long long L = m0 + m;
        bool valid = false;
        long long obase = 0;
        if (L < p.Mtot) {
          const uint32_t n = fdiv((uint32_t)L, p.fd_img);
          const uint32_t rem = (uint32_t)L - n * p.fd_img.d;
          const int e = (int)fdiv(rem, p.fd_WL);
          const int f = (int)rem - e * p.WL;
          const int oh = e * p.ph_step_h + p.ph_off_h[tc.ph];
          const int ow = f * p.ph_step_w + p.ph_off_w[tc.ph];
          valid = oh >= 0 && oh < p.Hd && ow >= 0 && ow < p.Wd;
          obase = (long long)n * p.dst_nstride + (long long)oh * p.Wd + ow;
        }
        const uint32_t tcol = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)((acc * p.MH + h) * p.NT);
        const int nbase = tc.nt * p.NT;
        const int nvalid = min(p.NT, p.Cd - nbase);  // output channels of this tile (NT is a multiple of 16)
        // 16-column chunks; the TMEM load of chunk i+1 is in flight while chunk i is stored.
        const int nchunk = (nvalid + 15) >> 4;
        uint32_t ra[16], rb[16];
        if (ntaps != 0) {
          tmem_ld16(tcol, ra);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) ra[j] = rb[j] = 0u;
        }
        const long long ostep = HdWd;
        if constexpr (EPI) {
          // Fused epilogue: the old values of up to EG = 2 16-channel chunks are all read before
          // the first of them is used (32 loads in flight per lane: the reads of the old output
          // are latency-bound otherwise), and so are the chunks' bias values, one per lane
          // (lane j holds channel j of a chunk; the warp broadcasts them with shuffles, so no
          // bias read waits behind an output store); then each chunk's accumulator columns are
          // loaded from TMEM, combined and stored.
          constexpr int EG = 2;
          for (int c0 = 0; c0 < nchunk; c0 += EG) {
            float old[EG][16], bsel[EG];
#pragma unroll
            for (int g = 0; g < EG; ++g) {
              const int ch = nbase + 16 * (c0 + g) + (lane & 15);
              bsel[g] = (p.bias != nullptr && 16 * (c0 + g) + (lane & 15) < nvalid) ? load_elem<DT>(p.bias, ch) : 0.f;
#pragma unroll
              for (int j = 0; j < 16; ++j) old[g][j] = 0.f;
            }
            if (valid && p.beta != 0.f) {
#pragma unroll
              for (int g = 0; g < EG; ++g) {
                const int ci = c0 + g;
                const long long ob = obase + (long long)(nbase + 16 * ci) * ostep;
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  if (ci < nchunk && 16 * ci + j < nvalid) old[g][j] = load_elem<DT>(p.dst, ob + j * ostep);
              }
            }
#pragma unroll
            for (int g = 0; g < EG; ++g) {
              const int ci = c0 + g;
              if (ci >= nchunk) break;
              if (ntaps != 0 && ci > 0) {
                tmem_ld16(tcol + (uint32_t)(16 * ci), ra);
                tmem_ld_wait();
              }
              float bv[16];  // the chunk's bias values in every lane (all lanes shuffle)
#pragma unroll
              for (int j = 0; j < 16; ++j) bv[j] = __shfl_sync(0xffffffffu, bsel[g], j);
              if (valid) {
                const long long ob = obase + (long long)(nbase + 16 * ci) * ostep;
                const int lim = nvalid - 16 * ci;
                store16_epi<DT>(p, ob, ostep, lim < 16 ? lim : 16, ra, old[g], bv);
              }
            }
          }
          continue;
        }
        for (int ci = 0; ci < nchunk; ci += 2) {
          const bool two = ci + 1 < nchunk;
          if (ntaps != 0 && two) tmem_ld16(tcol + (uint32_t)(16 * (ci + 1)), rb);
          if (valid) {
            const long long ob = obase + (long long)(nbase + 16 * ci) * ostep;
            const int lim = nvalid - 16 * ci;
            store16<DT, EPI>(p, ob, ostep, nbase + 16 * ci, lim < 16 ? lim : 16, ra);
          }
          if (ntaps != 0 && two) tmem_ld_wait();
          if (!two) break;
          if (ntaps != 0 && ci + 2 < nchunk) tmem_ld16(tcol + (uint32_t)(16 * (ci + 2)), ra);
          if (valid) {
            const long long ob = obase + (long long)(nbase + 16 * (ci + 1)) * ostep;
            const int lim = nvalid - 16 * (ci + 1);
            store16<DT, EPI>(p, ob, ostep, nbase + 16 * (ci + 1), lim < 16 ? lim : 16, rb);
          }
          if (ntaps != 0 && ci + 2 < nchunk) tmem_ld_wait();
        }
      }
      if (ntaps != 0) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_at(acce, acc));
        if (++acc == p.ACCB) {
          acc = 0;
          aphase ^= 1u;
        }
      }
    }
  } else {
    // =============================================================== MMA issuers
    // The whole warp runs the loop (warp-uniform control flow and descriptor arithmetic);
    // one elected lane issues the MMAs, with the taps' operand offsets read from the kernel
    // parameters, and commits.
    const int issuer = warp - kMmaWarp;  // accumulator half this warp owns
    if (issuer < nissuers) {
      const bool leader = elect_one();
      const uint32_t id = idesc(KIND, 128, p.NT, 0, 0);
      // Descriptor high halves (stride byte offset 128 B, version) are constant.
      const uint32_t d_hi = (uint32_t)(sdesc(0u, 0u, 128u) >> 32);
      const uint32_t a_ks = 2u * (uint32_t)rows, b_ks = 2u * (uint32_t)p.NT;
      long long counter = 0;
      int acc = 0;
      uint32_t aphase = 0;
      bool ok = true;
      bool issued_any = false;
      for (long long t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
        const TileCoord tc = decode_tile(p, t);
        const int ntaps = p.ph_ntaps[tc.ph];
        if (ntaps == 0) continue;
        const int tap0 = p.ph_tap_begin[tc.ph];
        if (!mbar_wait(bar_at(acce, acc), aphase ^ 1u, abort_flag, &g_tap_err)) break;
        tc_fence_after();
        const uint32_t dcol = tmem + (uint32_t)((acc * p.MH + issuer) * p.NT);
        for (int kb = 0; kb < p.nkb; ++kb, ++counter) {
          const int stage = (int)(counter % S);
          const uint32_t fphase = (uint32_t)((counter / S) & 1);
          if (!mbar_wait(bar_at(full, stage), fphase, abort_flag, &g_tap_err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // Low descriptor halves of this stage's operands (this issuer's 128 rows of A).
          const uint32_t a_st = a0 + (uint32_t)stage * p.a_stage_bytes + (uint32_t)issuer * 128u * 16u;
          const uint32_t b_lo0 = (uint32_t)sdesc(b0 + (uint32_t)stage * p.b_stage_bytes, (uint32_t)p.NT * 16u, 0u);
          // In tap-pair mode the A entry carries the chunk stride to the pair's second tap.
          const uint32_t a_lo0 = (uint32_t)sdesc(a_st, NCH >= 2 ? (uint32_t)rows * 16u : 0u, 0u);
          const bool first = kb == 0;
          if (leader) {
            switch (NCH) {
              case 1: issue_stage<KIND, 0>(p, tap0, ntaps, dcol, a_lo0, b_lo0, d_hi, id, a_ks, b_ks, first); break;
              case 2: issue_stage<KIND, 1>(p, tap0, ntaps, dcol, a_lo0, b_lo0, d_hi, id, a_ks, b_ks, first); break;
              case 4: issue_stage<KIND, 2>(p, tap0, ntaps, dcol, a_lo0, b_lo0, d_hi, id, a_ks, b_ks, first); break;
              case 8: issue_stage<KIND, 4>(p, tap0, ntaps, dcol, a_lo0, b_lo0, d_hi, id, a_ks, b_ks, first); break;
              default: issue_stage<KIND, 8>(p, tap0, ntaps, dcol, a_lo0, b_lo0, d_hi, id, a_ks, b_ks, first); break;
            }
          }
          __syncwarp();
          if (leader) tc_commit(bar_at(empty, stage));
          issued_any = true;
        }
        if (!ok) break;
        if (leader) tc_commit(bar_at(accf, acc));
        if (++acc == p.ACCB) {
          acc = 0;
          aphase ^= 1u;
        }
      }
      if (!ok && issued_any && leader) {
        // Wait (bounded) for every MMA this warp issued before TMEM is released.
        tc_commit(drain + 8u * (uint32_t)issuer);
        mbar_wait_drain(drain + 8u * (uint32_t)issuer, 0);
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

// ---------------------------------------------------------------------------- packing
// Filter pack alone (pack_filter_one per chunk).
template <int DT>
__global__ void __launch_bounds__(256) pack_filter_kernel(const __grid_constant__ PackPlan pp) {
  griddep_launch_dependents();  // the GEMM may start; it waits for this grid before reading wpack
  const int NCH = pp.CB / (DT == 0 ? 4 : 8);
  const uint32_t total = (uint32_t)pp.n_ntiles * pp.nkb * NCH * pp.NT * pp.ntaps_total;
  for (uint32_t idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += gridDim.x * blockDim.x)
    pack_filter_one<DT>(pp, idx);
}

// The two packs that precede a tap GEMM with packed-source staging, in one launch: blocks
// [0, xblocks) run the source's channel-chunk pack units, the others the filter chunks, so
// that neither waits for the other's tail.
template <int DT>
__global__ void __launch_bounds__(256) tap_packs_kernel(const __grid_constant__ NhwcPackPlan px,
                                                        const __grid_constant__ PackPlan pp, unsigned xblocks) {
  extern __shared__ __align__(16) uint8_t pk_smem[];
  griddep_launch_dependents();  // the GEMM may start; it waits for this grid before its copies
  if (blockIdx.x < xblocks) {
    for (uint32_t u = blockIdx.x; u < px.units; u += xblocks) nhwc_pack_unit<DT>(px, u, pk_smem);
  } else {
    const int NCH = pp.CB / (DT == 0 ? 4 : 8);
    const uint32_t total = (uint32_t)pp.n_ntiles * pp.nkb * NCH * pp.NT * pp.ntaps_total;
    const uint32_t nthr = (gridDim.x - xblocks) * blockDim.x;
    for (uint32_t idx = (blockIdx.x - xblocks) * blockDim.x + threadIdx.x; idx < total; idx += nthr)
      pack_filter_one<DT>(pp, idx);
  }
}

// ---------------------------------------------------------------------------- launchers
size_t tap_gemm_smem_bytes(const TapPlan& p) {
  size_t b = (size_t)p.stages * (p.a_stage_bytes + p.b_stage_bytes);
  b = (b + 15) & ~size_t(15);
  b += 8 * (2 * p.stages + 6) + 8 + 4 * p.stages + 16;
  return b + 1024;  // alignment slack for the dynamic base
}

static std::atomic<int> g_smem_set[2][2][kMaxDevices];

template <int DT, bool EPI>
cudaError_t launch_tap_gemm_t(const cudaLaunchConfig_t& cfg, const TapPlan& p, size_t smem) {
  const cudaError_t e = ensure_dyn_smem(tap_gemm_kernel<DT, EPI>, smem, g_smem_set[DT][EPI ? 1 : 0]);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, tap_gemm_kernel<DT, EPI>, p);
}

// Launched with programmatic stream serialization: the kernel's set-up overlaps the filter
// pack that precedes it in the stream (the producers wait for it before the first copy).
cudaError_t launch_tap_gemm(const TapPlan& p, int dt, int grid, cudaStream_t st) {
  const size_t smem = tap_gemm_smem_bytes(p);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool epi = p.bias != nullptr || p.beta != 0.f;
  cudaError_t e;
  if (dt == 0)
    e = epi ? launch_tap_gemm_t<0, true>(cfg, p, smem) : launch_tap_gemm_t<0, false>(cfg, p, smem);
  else
    e = epi ? launch_tap_gemm_t<1, true>(cfg, p, smem) : launch_tap_gemm_t<1, false>(cfg, p, smem);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Source pack px (units over at most 6 blocks per SM) and filter pack pp (one chunk per thread,
// at most 2 blocks per SM of threads) in one launch.
cudaError_t launch_tap_packs(const NhwcPackPlan& px, const PackPlan& pp, int dt, int num_sms, cudaStream_t st) {
  const int CHUNK = dt == 0 ? 4 : 8;
  const size_t smem = nhwc_pack_smem_bytes(px, dt);
  const long long per_sm = std::max<long long>(1, std::min<long long>(6, (long long)(200 * 1024) / (long long)std::max<size_t>(smem, 1)));
  const long long xb = std::max(1ll, std::min<long long>((long long)px.units, (long long)num_sms * per_sm));
  const long long total = (long long)pp.n_ntiles * pp.nkb * pp.ntaps_total * (pp.CB / CHUNK) * pp.NT;
  const long long fb = std::max(1ll, std::min<long long>((total + 255) / 256, (long long)num_sms * 2));
  static std::atomic<int> set_bytes[2][kMaxDevices];
  cudaError_t e;
  if (dt == 0) {
    e = ensure_dyn_smem(tap_packs_kernel<0>, smem, set_bytes[0]);
    if (e != cudaSuccess) return e;
    tap_packs_kernel<0><<<(unsigned)(xb + fb), 256, smem, st>>>(px, pp, (unsigned)xb);
  } else {
    e = ensure_dyn_smem(tap_packs_kernel<1>, smem, set_bytes[1]);
    if (e != cudaSuccess) return e;
    tap_packs_kernel<1><<<(unsigned)(xb + fb), 256, smem, st>>>(px, pp, (unsigned)xb);
  }
  return cudaGetLastError();
}

cudaError_t launch_pack_filter(const PackPlan& pp, int dt, cudaStream_t st) {
  const int CHUNK = dt == 0 ? 4 : 8;
  const long long total = (long long)pp.n_ntiles * pp.nkb * pp.ntaps_total * (pp.CB / CHUNK) * pp.NT;
  const long long blocks = std::max(1ll, std::min<long long>((total + 255) / 256, 8192));
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

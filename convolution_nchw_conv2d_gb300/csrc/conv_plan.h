// conv_plan.h -- launch plans shared by the host planner (conv2d_api.cpp) and the
// kernels.  Plain structs of integers and pointers, passed by value as kernel
// parameters.
//
// Every op is run as an implicit GEMM over a "linear position space": positions
// L = n*EL*WL + e*WL + f enumerate an EL x WL grid per image, laid out row after row.
// A filter tap then reads the source at L + off, one constant per tap, so one
// staged tile of source rows serves every tap of the filter by a row offset.
// Positions with no output (f beyond the output width, e beyond the output height)
// are computed and discarded.  For stride > 1 the source is split into
// stride_h*stride_w phase planes (forward, backward-filter) or the output is split
// into phases (backward-data), so that every tap is a unit-stride shift.
#pragma once
#include <cstdint>

#include <cuda.h>  // CUtensorMap (the plan only carries it; encoding is done by the host planner)

namespace cg3 {

// Device-side error codes a kernel records in its error word (read back by conv2d_device_status):
// a bounded pipeline wait that expired, or a shared-memory carve-up larger than the launch gave.
enum : int { DEV_ERR_NONE = 0, DEV_ERR_TIMEOUT = 1, DEV_ERR_LAYOUT = 2 };

// Unsigned 32-bit division by a divisor fixed at planning time, as a multiply-high and
// shifts (Granlund and Montgomery, "Division by Invariant Integers using
// Multiplication", PLDI 1994, unsigned case): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1,  n / d = (t + ((n - t) >> min(l,1))) >> max(l-1,0)
// where t = mulhi(m, n), exact for every n < 2^32.
struct FastDiv {
  uint32_t d, m, s1, s2;
};

inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  uint32_t l = 0;
  while (l < 32 && (1ull << l) < d) ++l;
  f.d = d;
  f.m = (uint32_t)((((1ull << 32) * ((1ull << l) - d)) / d) + 1);
  f.s1 = l < 1 ? l : 1;
  f.s2 = l > 1 ? l - 1 : 0;
  return f;
}

#ifdef __CUDACC__
__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
  const uint32_t t = __umulhi(n, f.m);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}
#endif

constexpr int kMaxPlanes = 64;   // stride_h * stride_w
constexpr int kMaxPhases = 64;
constexpr int kMaxTaps = 256;    // R * S of one pass (forward / backward-data split larger filters into passes)

// Forward and backward-data: D[position, out_channel] = sum over taps and source
// channels of S[channel, position + tap_off] * Wpacked[tap, out_channel, channel].
struct TapPlan {
  // Source planes packed channel-chunk-wise ([plane][chunk][position L][16 bytes]: CHUNK
  // consecutive channels of the plane's pixel at L, zero outside the tensor) as a 3-D tensor
  // of 8-byte elements (2*L, chunk, plane); valid when a_tma.  A stage's staged rows of one
  // plane and chunk are then one contiguous run, loaded by tensor copies of a_box rows (the
  // rows past the last position read as zero).
  CUtensorMap tm_src;
  int a_tma;             // 1: staged rows come from tm_src (rows = a_nbox * a_box)
  int a_box, a_nbox;
  int a_one;             // 1 (rows <= 256): tm_src views the planes as (2, L, chunk, plane) and
                         // one copy of box (2, rows, NCH, planes of the stage) stages them all;
                         // 0: one copy per (plane, chunk, box of a_box rows) of the view above
  int plane_per_phase;   // 1 (with a_tma, one plane): phase ph reads the plane shifted by
                         // ph_shift[ph] positions, so a stage holds the tile's phase window alone
  int ph_shift[kMaxPhases];
  const void* src;       // x (forward) or dy (backward-data), NCHW
  void* dst;             // y or dx, NCHW
  const void* bias;      // optional, one value per destination channel (NULL: none)
  long long src_nstride, dst_nstride;  // elements from one image to the next (C*H*W unless
                                       // the tensors hold several groups)
  float beta;            // dst = D + bias + beta * dst (beta 0: dst is not read)
  const void* wpack;     // packed filter, see pack layout in conv_tap_gemm.cu
  int N, Cs, Hs, Ws;     // source tensor
  int Cd, Hd, Wd;        // destination tensor
  int WL, EL;            // linear-space row width and rows per image
  long long Mtot;        // N * EL * WL (< 2^31)
  FastDiv fd_img, fd_WL; // division by EL*WL and by WL
  int n_mtiles, n_ntiles, nkb;  // tiles along positions / out channels; channel blocks
  long long total_tiles;        // nph * n_mtiles * n_ntiles
  int rows;              // staged source rows per plane (multiple of 8)
  int npl;               // source planes
  int pl_step_h, pl_step_w;
  int pl_off_h[kMaxPlanes], pl_off_w[kMaxPlanes];
  int nph;               // output phases
  int ph_step_h, ph_step_w;
  int ph_off_h[kMaxPhases], ph_off_w[kMaxPhases];
  int ph_tap_begin[kMaxPhases], ph_ntaps[kMaxPhases];
  int max_taps_ph;       // B stage region holds this many taps
  int ntaps_total;
  int tap_plane[kMaxTaps];
  int tap_off[kMaxTaps];
  // MMA operand offsets of tap t within a stage, in 16-byte units: tap_a = A rows (plane * NCH *
  // rows + tap_off; in tap-pair mode, NCH = 1, the pair's first tap also carries the chunk stride
  // to its second tap in bits 16..29, the descriptor's leading-byte-offset field), tap_b = B
  // (index within the phase * NCH * NT).  Filled once the tile shape is chosen.
  int tap_a[kMaxTaps], tap_b[kMaxTaps];
  int stages;
  int MH;                // 128-row halves per tile (1 or 2)
  int NT;                // GEMM N per tile (multiple of 16, <= 256)
  int CB;                // source channels per pipeline stage (multiple of 2 chunks)
  int ACCB;              // TMEM accumulator buffers (1 or 2)
  int a_stage_bytes, b_stage_bytes;
  int tmem_cols;
};

// Filter packing for TapPlan: one 16-byte chunk per (n_tile, k_block, tap, chunk, row).
struct PackPlan {
  const void* w;          // KCRS filter
  void* wpack;
  int K, C, R, S;         // filter dims as stored
  int transpose;          // 0: out channel = K index, source channel = C index (forward)
                          // 1: out channel = C index, source channel = K index (backward-data)
  int Cd, Cs;             // GEMM N extent and source-channel extent
  int n_ntiles, nkb, ntaps_total;
  int NT, CB;
  int tap_r[kMaxTaps], tap_s[kMaxTaps];
  int flip;               // convolution mode: tap (r, s) reads w[.., R-1-r, S-1-s]
  // Grouped filter packed block-diagonally (gd != 0): gs source and gd out channels per group;
  // an element whose source and out channel lie in different groups is zero, and C is the
  // filter's channels per group.
  int gs, gd;
};

// Backward-filter as one implicit GEMM per tile:
//   D[m, k] = sum over positions L of X_plane(tap)[c, L + tap_off[tap]] * dy[k, L]
// over the forward linear position space (dy is zero where a position has no output),
// with each row m standing for one (channel c, filter tap) pair.  Rows come in units of
// 32 (one TMEM lane quarter): for C >= 32 a unit is 32 consecutive channels of one tap,
// for C < 32 a unit is TPU taps x C channels (lane l: c = l mod C, tap = first + l / C).
// Units are ordered channel group by channel group, taps within a group; a tile is 4
// units (128 rows) x NK output channels x one range of positions (split-K).
//
// The A operand (the im2col of x for the tile's rows, 32 TMEM columns at a time) is
// written into TMEM by builder warps from a ring of staged x; B = dy[k, L] is K-major
// (positions contiguous, as in NCHW) in shared memory.  The ring is [plane][channel][xs]:
// slot (q + sigma) mod rlen of a row holds tile-relative position q of that plane and
// channel, and every position is loaded once per tile.  sigma aligns 16-byte slot groups
// with 16-byte pixel groups, which are copied with 16-byte cp.async; the row stride xs is
// 16 bytes more than a multiple of 128, so the builders' 16-byte reads of 8 channel rows
// at the same slot fall in distinct banks.  Split partials [split][tap][C][K] (fp32) are
// added in a fixed order by a second kernel.
struct WgradPlan {
  // dy as a 4-D tensor (w, k, row e, image n) for copy-engine loads of one 16-byte chunk of
  // positions for NK output channels ([k][CHUNK] in shared memory); valid when use_tma.
  CUtensorMap tm_dy;
  // x as a 4-D tensor (w, h, c, n) with a box of one image row (WL pixels from column
  // -align(pad_w)) by 32 channels; valid when use_tma.
  CUtensorMap tm_x;
  // dy as a 5-D tensor (w mod CHUNK, k, w / CHUNK, row e, image n) for copy-engine loads of
  // one whole linear row of positions for NK output channels, [chunk][k][CHUNK] in shared
  // memory; valid when TRU > 1.
  CUtensorMap tm_dyr;
  int use_tma;           // copy-engine staging (unit column stride, aligned tensors): dy by
                         // tensor copies, x by tensor copies of whole rows into a row ring
  // Row ring (use_tma): [NR row slots][plane][xr channel rows][WL].  Position L lives at
  // slot s = L + delta: row slot (s / WL) mod NR, column s mod WL; the copy of linear row R
  // holds pixels -align(pad_w) .. +WL-1 of its image row, so columns past the image and
  // before it read as zeros.  WL = CHUNK mod 2 CHUNK keeps 16-byte reads of 8 consecutive
  // channel rows in distinct banks.
  int NR, xr, delta;
  FastDiv fd_NR;
  int WLx;               // row ring pitch of one channel row (elements, >= WL)
  // Row-tap sharing (TRU > 1, row ring only): a unit is 32 channels x one base tap
  // (r0, s) and stands for the TRU taps (r0 + j, s), j < TRU.  Since tap (r0 + j, s) reads
  // x at L + j*WL + off(r0, s), the sum over positions L equals the sum over L' = L + j*WL of
  // x[L' + off(r0, s)] * dy[L' - j*WL]: one A operand built from x at L' serves all TRU taps,
  // each paired with dy shifted back by j linear rows (j*dil_h rows with row dilation: the
  // shift is j*tru_step).  dy is then staged as a ring of NRd whole linear rows,
  // [row slot][chunk][k][CHUNK], and the positions L' run over [0, Mtot + (TRU-1)*tru_step*WL)
  // (dy reads as zero outside [0, Mtot)).
  int TRU;               // row taps per unit (1: every unit is one tap)
  int tru_step;          // linear rows between consecutive row taps (the row dilation)
  int NRd;               // dy ring rows (TRU > 1)
  FastDiv fd_NRd;
  long long Mit;         // positions iterated (Mtot + (TRU - 1) * tru_step * WL)
  int unit_tap[kMaxTaps];  // base tap of the j-th unit of a channel group (TPU == 1)
  const void* x;         // NCHW
  const void* dy;        // N K P Q
  long long x_nstride, dy_nstride;  // elements from one image to the next (C*H*W and K*P*Q
                                    // unless the tensors hold several groups)
  float* partial;        // [split][R*S][C][K] fp32
  int N, C, H, W, K, P, Q;
  int R, S, RS;
  int WL, EL;
  long long Mtot;        // positions (< 2^31)
  FastDiv fd_img, fd_WL; // division by EL*WL and by WL
  FastDiv fd_EL, fd_rlen;  // division by EL and by rlen
  int npl;
  int pl_step_h, pl_step_w;
  int pl_off_h[kMaxPlanes], pl_off_w[kMaxPlanes];
  int tap_plane[kMaxTaps], tap_off[kMaxTaps];  // per filter tap r*S + s
  int tap_rc[kMaxTaps];  // tap_off as (linear rows << 16) | columns
  int max_off;           // largest tap_off
  int Cg, TPU, upc;      // channels per unit, taps per unit, units per channel group
  FastDiv fd_upc;        // division by upc
  int nunits;            // units of 32 rows in all
  int n_mtiles, n_ntiles, nsplit;
  int G;                 // m-tiles per CTA tile (one TMEM accumulator each; x and dy staged once)
  int n_mgroups;         // ceil(n_mtiles / G)
  long long split_len;   // positions per split (multiple of KB)
  long long total_tiles; // n_mgroups * n_ntiles * nsplit
  int NK;                // output channels k per tile (MMA N, multiple of 16, <= 256)
  int KB;                // positions per pipeline stage (multiple of 32 TMEM columns)
  int stages;
  int xch;               // channels staged per tile (span of the widest tile)
  int xs;                // ring row stride in elements (>= rlen)
  int rlen;              // ring slots per row (multiple of 32)
  int sigma;             // slot of tile-relative position q is (q + sigma) mod rlen
  int vec_x;             // 16-byte x loads allowed (unit column stride, aligned rows)
  int a_stage_bytes;     // dy tile bytes per stage
  int accb;              // TMEM accumulator sets of G tiles (1 or 2)
  int tmem_cols;
  int vec_dy;            // 16-byte dy copies allowed (alignment / contiguity)
};

// Sum of the split partials [split][rows][K] of the channel-chunked backward-filter, transposed:
// dw[k][row] = sum over splits of partial[split][row][k] (+ beta * dw), row = c*R*S + r*S + s
// (convolution mode writes tap r*S + s at (R-1-r)*S + S-1-s).
struct ReduceTPlan {
  const float* partial;
  void* dw;
  int rows, K, RS, nsplit;
  float beta;
  int flip;
  // Grouped filter from the whole problem's partials (gk != 0): gk output and gc input channels
  // per group; only the diagonal blocks (c / gc == k / gk) are kept, dw is K x gc x R x S.
  int gk, gc;
};

struct ReducePlan {
  const float* partial;
  void* dw;              // K x C x R_out x S_out, fp32 or bf16
  int K, C, R, S;        // the partials' filter: R x S taps
  int nsplit, k_pad, c_pad;
  float beta;            // dw = sum + beta * dw (beta 0: dw is not read)
  int flip;              // convolution mode: the placed tap (r, s) is dw[.., R_out-1-r, S_out-1-s]
  // Placement of partial tap (r', s') in dw: (r0 + rstep * r', s0 + sstep * s') of an
  // R_out x S_out filter (one stride phase of a strided filter; the identity otherwise).
  int R_out, S_out, r0, s0, rstep, sstep;
  // Grouped filter from the whole problem's partials (gk != 0): gk output and gc input channels
  // per group; only the diagonal blocks (c / gc == k / gk) are kept, dw is K x gc x R_out x S_out.
  int gk, gc;
};

// Channel-chunked, zero-padded planes of an NCHW tensor ("NHWC within chunks"):
//   dst[pl][cc][n][e][f][j] = src[n][CHUNK*cc + j][e*step_h + off_h[pl]][f*step_w + off_w[pl]]
// for e < EX, f < WL, j < CHUNK (CHUNK = 16 bytes of elements), zero where the channel, row or
// column lies outside the source.  Every 16-byte group holds CHUNK consecutive channels of one
// position, so a tile of positions x channel chunks is one tensor copy into the MN-major operand
// layout, and a shift of the position by one is a shift of one 16-byte row.
//
// Work unit = (image n, group of cg chunks, tile of te padded rows e): the source rows that the
// tile's planes read, [h_lo, h_lo + span] with h_lo = e0*step_h + off_h_min, are one contiguous
// run per channel, staged in shared memory by coalesced copies; the unit's output of each chunk
// and plane is one contiguous run of te*WL 16-byte groups.
struct NhwcPackPlan {
  const void* src;
  void* dst;
  long long src_nstride;  // elements from one source image to the next
  int N, C, H, W;         // source extents (C channels per image)
  int nchunk;             // ceil(C / CHUNK)
  int EX, WL;             // padded plane extent
  FastDiv fd_WL;          // division by WL
  int npl;                // planes
  int step_h, step_w;
  int off_h[kMaxPlanes], off_w[kMaxPlanes];
  int off_h_min, h_span;  // smallest plane row offset; largest minus smallest
  int te, n_etiles;       // padded rows per unit; row tiles per image
  int cg, ngroups;        // chunks per unit; chunk groups per image
  int ch_pitch;           // staged elements per channel: (te-1)*step_h + h_span + 1 rows of W,
                          // rounded up to 16 bytes
  unsigned units;         // N * ngroups * n_etiles (< 2^31)
  FastDiv fd_et, fd_ng;   // division by n_etiles and by ngroups
};

// Backward-filter on channel-chunked planes (bf16): for every filter tap t of a stride phase,
//   D_t[c, k] = sum over positions L of Xq_plane(t)[c, L + off_t] * DYq[k, L]
// over the padded position space L = n*EX*WL + e*WL + f shared by all phases (DYq is zero past
// the output rows and columns).  Both operands are MN-major tiles in shared memory (16 bytes =
// 8 channels of one position), so every tap is a row offset of the staged x tile.  A tile is
// (tap group, 128 channels, NK output channels, one range of positions); a tap group is up to T
// taps of one phase, sorted by offset, staged as one x tile spanning their offsets.  Split
// partials [split][C*R*S][K] (fp32, row c*R*S + r*S + s) are added by a fixed-order reduce that
// transposes them into KCRS.  The tensor maps view the packed planes as 8-byte elements (two per
// position), so that each copy row is a contiguous run of positions, not one 16-byte group.
struct WgradMnPlan {
  CUtensorMap tm_x;   // Xq as (2*positions, C/8, planes) of 8-byte elements, box (2*KBX, 16, 1)
  CUtensorMap tm_dy;  // DYq as (2*positions, K/8), box (2*KB, NK/8)
  float* partial;
  int C, K, RS;
  long long Mtot;     // positions N*EX*WL
  int KB, KBX, stages, NK, T;
  int n_ctiles, n_ktiles, ngroups, nsplit;
  long long split_len;   // positions per split (multiple of KB)
  long long total_tiles; // nsplit * ngroups * n_ctiles * n_ktiles
  int a_stage_bytes, b_stage_bytes;  // stage strides (1024-byte multiples)
  int tx_bytes;                      // bytes of one stage's two boxes
  int tmem_cols;
  // tap group g: plane, first tap index, tap count, position offset of the staged x tile
  int grp_plane[kMaxTaps], grp_tap0[kMaxTaps], grp_ntaps[kMaxTaps], grp_off0[kMaxTaps];
  // tap i: row offset in the staged x tile, and its filter tap r*S + s (the partial's slot)
  int tap_delta[kMaxTaps], tap_out[kMaxTaps];
};

// Backward-data for few input channels (C <= 8).  With output row phase phi_h (h = p*sh - ph +
// phi_h) the filter rows r that reach dx row h from dy row p - d are those with
// r*dh = d*sh + phi_h, so
//     T[(p, q), (c, phi_h, s)] = sum over d, k of dy[k, p - d, q] * w[k, c, (d*sh + phi_h)/dh, s]
// is a GEMM over k for every row shift d (one MMA set per shift: the shift is a whole-row
// offset of the staged dy operand), and dx[c, p*sh - ph + phi_h, q*sw - pw + phi_w] is the
// sum of T over the taps s that land on column phase phi_w, from columns q - (s*dw - phi_w)/sw
// (a warp-shuffle fold).  A tile owns 8 dy "anchor" rows x (32 - dlt_w) columns and stages
// dy rows p_lo - dlt_h .. p_lo + 7 and columns q_lo .. q_lo + 31.  Layouts: dy NKPQ, w KCRS,
// dx NCHW.
struct C2iPlan {
  CUtensorMap tm_dy;  // dy (Q, P, K, N) fp32, box (36, EH, 16, 1); valid when use_tma
  int use_tma;        // dy boxes by tensor copies (else the builders read global memory)
  int nraw;           // dy box slots in shared memory (0 without tensor copies)
  int nraw_tma;       // the slots a launch with tensor copies uses
  const void* dy;
  const void* w;
  const void* bias;   // per c, or NULL
  void* dx;
  float beta;         // dx = sum + bias + beta * dx
  int flip;           // convolution mode: the filter rotated by 180 degrees
  int N, C, H, W, K, R, S, P, Q;
  int sh, sw, ph, pw, dh, dw;
  long long dy_nstride, dx_nstride;  // elements from one image to the next
  int Nr;             // MMA N: C*sh*8 ((c, phi_h, s), s padded to 8) rounded up to 16
  int nkb;            // blocks of 16 dy channels (K padded with zeros)
  int dlt_h, dlt_w;   // largest row shift floor((R-1)*dh/sh), column shift floor((S-1)*dw/sw)
  int EH;             // staged dy rows: 8 + dlt_h
  int TWq;            // owned dy columns per tile: 32 - dlt_w
  int p_start, q_start;  // first anchor dy row / owned column of tile 0: floor(ph/sh), floor(pw/sw)
  int ntp, ntq;       // tiles per image along dy rows (8 anchors) / columns (TWq)
  long long tiles;    // N * ntp * ntq
  int b_bytes;        // filter operand: (dlt_h+1) shifts x (nkb*4) chunks x Nr rows x 16 bytes
  int a_bytes;        // one staged operand: 4 chunks x EH*32 rows x 16 bytes
  int nast;           // staged operand slots
  int tmem_cols;      // two accumulators of 2 x Nr columns
};

// Space-to-depth of x for strided backward-filter: xs[n][a*sw + b][c][i][j] =
// x[n][c][i*sh + a][j*sw + b] (zero where that lies outside x), i < Hp, j < Wp.
struct S2dPlan {
  const void* x;
  void* xs;
  int N, C, H, W, sh, sw, Hp, Wp;
};

// Per-channel sum of an NCHW-like tensor t (N, Ch, HW): out[ch] = sum_{n, i} t[n, ch, i]
// (+ beta * out[ch]), as fixed-order partials part[ch * N + n] and a final pass.
struct ChanSumPlan {
  const void* t;
  void* out;
  float* part;           // Ch * nblk fp32 (workspace)
  int N, Ch;
  long long HW;
  float beta;
  int ipb, nblk;         // images per block; blocks per channel = ceil(N / ipb)
};

// Depthwise layers (one input channel per group: groups == C, M = K / C output channels per
// input channel), all three ops on CUDA cores, direct form:
//   forward        y[n, k, p, q]  = sum_{r,s} x[n, k / M, p*sh - ph + r*dh, q*sw - pw + s*dw] * w[k, r', s']
//   backward-data  dx[n, c, h, w] = sum_{m < M} sum_{r,s} dy[n, c*M + m, p, q] * w[c*M + m, r', s']
//                                   over the (r, s) with h + ph - r*dh = p*sh, w + pw - s*dw = q*sw
//   backward-filter dw[k, r', s'] = sum_{n,p,q} x[n, k / M, p*sh - ph + r*dh, ...] * dy[n, k, p, q]
// with (r', s') = (r, s), or (R-1-r, S-1-s) in convolution mode; fp32 sums in a fixed order.  The
// filter gradient sums split partials [split][K][R*S] (a split: a range of images) in split
// order.
struct DwPlan {
  const void* x;
  const void* w;
  const void* dy;
  void* out;             // y, dx or dw
  const void* bias;      // per k (forward) or per c (backward-data), or NULL
  float beta;            // out = sum + bias + beta * out (beta 0: out is not read)
  int flip;
  int N, C, H, W, K, R, S, P, Q;
  int ph, pw, sh, sw, dh, dw;
  int M;                 // K / C
  float* partial;        // filter gradient: nsplit * K * R * S fp32 (workspace)
  int nsplit;            // filter gradient: image ranges of n_per_split images
  int n_per_split;
};

}  // namespace cg3

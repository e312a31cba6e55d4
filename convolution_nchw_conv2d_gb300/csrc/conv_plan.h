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

namespace cg3 {

constexpr int kMaxPlanes = 16;   // stride_h * stride_w
constexpr int kMaxPhases = 16;
constexpr int kMaxTaps = 256;    // R * S
constexpr int kMaxSlots = 64;    // (plane, residue) x copies staged by fp32 backward-filter

// Forward and backward-data: D[position, out_channel] = sum over taps and source
// channels of S[channel, position + tap_off] * Wpacked[tap, out_channel, channel].
struct TapPlan {
  const void* src;       // x (forward) or dy (backward-data), NCHW
  void* dst;             // y or dx, NCHW
  const void* wpack;     // packed filter, see pack layout in conv_tap_gemm.cu
  int N, Cs, Hs, Ws;     // source tensor
  int Cd, Hd, Wd;        // destination tensor
  int WL, EL;            // linear-space row width and rows per image
  long long Mtot;        // N * EL * WL
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
  int stages;
  int MH;                // 128-row halves per tile (1 or 2)
  int NT;                // GEMM N per tile (multiple of 16, <= 256)
  int CB;                // source channels per pipeline stage (multiple of 2 chunks)
  int ACCB;              // TMEM accumulator buffers (1 or 2)
  int a_stage_bytes, b_stage_bytes;
  int tmem_cols;
  int vec;               // source rows may be read with 16-byte loads (see stage_pixel_rows)
  int vec_phase[kMaxPlanes];
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
};

// Backward-filter: per tap t, D_t[k, c] = sum over positions L of
// dy[k, L] * Xplane(t)[c, L + tap_off[t]], split over position ranges.
// Taps are processed in groups (one group per CTA tile, the group's accumulators
// side by side in TMEM); tap t of the plan is filter tap tap_id[t] = r*S + s.
// bf16 stages x once per plane with positions along rows (an MN-major operand) and
// reaches tap t by the row offset tap_off[t].  tf32 operands must be K-major, where
// a 16-byte chunk holds 4 consecutive positions, so fp32 stages, per group, one copy
// of x per (plane, offset mod 4) "slot", shifted by that residue and starting at
// position 4*tg_qmin[g]; tap t is chunk offset tap_q[t] (relative to tg_qmin) of
// slot tap_slot[t] (an index into slot_plane/slot_res).  WL is a multiple of 4 and
// groups are formed per filter row offset, so a group's halo is a few positions.
struct WgradPlan {
  const void* x;         // NCHW
  const void* dy;        // N K P Q
  float* partial;        // [split][R*S][c_pad][k_pad] fp32
  int N, C, H, W, K, P, Q;
  int WL, EL;
  long long Mtot;
  int npl;
  int pl_step_h, pl_step_w;
  int pl_off_h[kMaxPlanes], pl_off_w[kMaxPlanes];
  int ntaps;
  int tap_id[kMaxTaps];
  int tap_plane[kMaxTaps], tap_off[kMaxTaps];   // bf16
  int tap_slot[kMaxTaps], tap_q[kMaxTaps];      // fp32
  int nslots;
  int slot_plane[kMaxSlots], slot_res[kMaxSlots];
  int slot_base[kMaxSlots];        // fp32: residue-0 slot of the same plane and group
  int slot_chunks;                 // fp32: chunks staged per slot (nchunks + 1)
  int x_shift;                     // fp32: staged x origin offset (aligns chunk starts)
  int n_tgroups;
  int tg_begin[kMaxTaps], tg_count[kMaxTaps];
  int tg_qmin[kMaxTaps], tg_slot_begin[kMaxTaps], tg_nslots[kMaxTaps];
  int nchunks;           // fp32: position chunks staged per slot per stage
  int n_ktiles, n_ctiles, nsplit;
  long long split_len;   // positions per split (multiple of the stage length)
  int rows;              // staged x rows per plane per stage (multiple of 8)
  int k_pad, c_pad;      // extents of the partial buffer
  long long total_tiles; // n_ktiles * n_ctiles * n_tgroups * nsplit
  int stages;
  int NC;                // channels per tile (GEMM N per tap, multiple of 16)
  int KB;                // positions per pipeline stage
  int a_stage_bytes, b_stage_bytes;
  int tmem_cols;
  int vec_dy;            // dy chunks may be copied with 16-byte cp.async
  int vec_x;             // x rows may be read with 16-byte loads
  int vec_phase[kMaxPlanes];  // bf16 x: see stage_pixel_rows
};

struct ReducePlan {
  const float* partial;
  void* dw;              // KCRS, fp32 or bf16
  int K, C, R, S;
  int nsplit, k_pad, c_pad;
};

}  // namespace cg3

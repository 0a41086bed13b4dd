// Activation staging of a routed batch ("NVFP4 MegaMoE Debug Log", section
// "NVFP4 MoE Pipeline": stage_activation; "NVFP4-1.1 Approach, Part 2": the
// padded per-expert layout), as device functions shared by the routing launch
// (route.cu) and by the side warps of the CTA-pair BF16 GEMM (gemm_pair.cu),
// which stage a later batch while the L2 GEMM of an earlier one runs.
//
// x is quantised once per token (PLAIN, per 16 along H) and the bytes are
// written into each of the token's k permuted rows.  The work comes in
// 1024-column segments of one token: lane i of a warp takes columns 32i..32i+31
// (two 16-blocks), so a warp's 16-byte nibble stores cover 512 contiguous bytes
// of each row, and a lane pair's four scale bytes form one word of the swizzled
// layout.  H % 64 == 0, so a lane pair is wholly inside the row or wholly past it.
//
// The padding rows [offsets[e] + counts[e], offsets[e+1]) of expert e (at most
// 127 rows, all inside the group's last 128-row band) get zero scale words and
// no nibbles: a zero E4M3 scale dequantises every E2M1 code (which has no NaN or
// infinity) to zero, so a padding row is an exact zero row of the GEMM whatever
// its nibbles hold.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

// Zero the padding scales of expert e: work items first, first + stride, ... of
// the band's H/64 x 32 items.  In a band's scale atom (512 bytes per 64
// columns), 16-byte line l holds the words of rows l, l+32, l+64, l+96; item
// (k4, l) zeroes the line with one 16-byte store when all four rows are
// padding, else the words of its padding rows (real rows' words are never
// touched, so this may run concurrently with the rows' own stores).
__device__ __forceinline__ void stage_padding(const StageJob& s, int e, int64_t first, int64_t stride) {
  const int64_t lo = __ldg(s.offsets + e) + __ldg(s.counts + e);
  const int64_t hi = __ldg(s.offsets + e + 1);
  if (hi <= lo) return;
  const int64_t band = (hi - 1) >> 7;
  if (hi > s.rows_max) {                                      // the group's band lies past a_sf
    if (first == 0) raise_error(s.err, kErrBounds);
    return;
  }
  const int first_pad = static_cast<int>(lo - band * 128);    // band-relative first padding row (1..127)
  const int k4_total = s.H / 64;
  const int64_t items = static_cast<int64_t>(k4_total) * 32;
  for (int64_t i = first; i < items; i += stride) {
    const int l = static_cast<int>(i & 31);
    const int64_t k4 = i >> 5;
    uint8_t* line = s.a_sf + (band * k4_total + k4) * 512 + l * 16;
    if (l >= first_pad) {
      *reinterpret_cast<uint4*>(line) = make_uint4(0, 0, 0, 0);
    } else {
#pragma unroll
      for (int c = 1; c < 4; ++c)
        if (l + 32 * c >= first_pad) *reinterpret_cast<uint32_t*>(line + 4 * c) = 0u;
    }
  }
}

// One lane's 32 values (two 16-blocks, four 16-byte BF16 loads in raw) ->
// their 16 bytes of nibbles and the two blocks' scale codes (byte q for block
// q); with a two-level scale the values quantised are fp32(x * g).
__device__ __forceinline__ void stage_quantize(const uint4 (&raw)[4], bool scaled, float g, uint4& nib,
                                               uint32_t& codes) {
  uint32_t w[4];
  codes = 0;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    float lo[8], hi[8];
    bf16x8_to_f32(raw[2 * q], lo);
    bf16x8_to_f32(raw[2 * q + 1], hi);
    if (scaled) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        lo[i] *= g;
        hi[i] *= g;
      }
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fmaxf(fabsf(lo[i]), fabsf(hi[i])));
    const BlockScale bs = block_scale(amax);
    w[2 * q] = quantize8(lo, bs);
    w[2 * q + 1] = quantize8(hi, bs);
    codes |= bs.code << (8 * q);
  }
  nib = make_uint4(w[0], w[1], w[2], w[3]);
}

// One warp's batch of segments item[0..kNS) (item = token * segs + segment,
// segs = ceil(H / 1024); item < 0: none) with its loads: each segment's x
// (2 KiB) and its token's k row indices (lane j loads slot j; k <= 32, broadcast
// later by shuffle), so a warp never waits on one index load per row.
template <int kNS>
struct StageBatch {
  int64_t item[kNS];
  int64_t tok[kNS];
  int64_t c0[kNS];          // this lane's first column; >= H: inactive lane or no item
  int32_t rows[kNS];
  uint4 raw[kNS][4];
};

// Issue the batch's loads (item[] set by the caller, warp-uniform).
template <int kNS>
__device__ __forceinline__ void stage_load(const StageJob& s, StageBatch<kNS>& b, int lane) {
  const int64_t segs = (s.H + 1023) / 1024;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(s.x);
#pragma unroll
  for (int n = 0; n < kNS; ++n) {
    b.tok[n] = b.item[n] >= 0 ? b.item[n] / segs : 0;
    b.c0[n] = b.item[n] >= 0 ? (b.item[n] - b.tok[n] * segs) * 1024 + lane * 32 : s.H;
    b.rows[n] = b.item[n] >= 0 && lane < s.k ? __ldg(s.inv_perm + b.tok[n] * s.k + lane) : 0;
    if (b.c0[n] < s.H) {
      const uint4* src = reinterpret_cast<const uint4*>(x + b.tok[n] * s.H + b.c0[n]);
#pragma unroll
      for (int i = 0; i < 4; ++i) b.raw[n][i] = __ldg(src + i);
    }
  }
}

// Quantise the batch's segments and write them into their k rows.  The whole
// warp takes part (the scale words are paired, the row indices broadcast, by
// shuffle).  A row index outside [0, rows_max) is not written and sets
// kErrBounds (the x_q row, which needs no index, still is).
template <int kNS>
__device__ __forceinline__ void stage_store(const StageJob& s, const StageBatch<kNS>& b, int lane) {
  const float g = s.x_gscale != nullptr ? __ldg(s.x_gscale) : 1.0f;
  const uint32_t k4_total = static_cast<uint32_t>(s.H / 64);
#pragma unroll
  for (int n = 0; n < kNS; ++n) {
    if (b.item[n] < 0) continue;             // warp-uniform
    const bool active = b.c0[n] < s.H;
    uint4 nib = make_uint4(0, 0, 0, 0);
    uint32_t codes = 0;
    if (active) stage_quantize(b.raw[n], s.x_gscale != nullptr, g, nib, codes);
    // lanes 2m, 2m+1 own one 64-column group: codes of its four blocks in order
    const uint32_t word = codes | (__shfl_down_sync(0xFFFFFFFFu, codes, 1) << 16);
    const uint32_t k4 = static_cast<uint32_t>(b.c0[n] / 64);
    const int64_t t = b.tok[n];
    // token-order rows (read by a gathering L1) and / or the permuted copies; the
    // scale words always go to the permuted, padded layout
    if (active && s.x_q != nullptr) *reinterpret_cast<uint4*>(s.x_q + t * (s.H / 2) + b.c0[n] / 2) = nib;
    for (int j = 0; j < s.k; ++j) {
      const int64_t r = __shfl_sync(0xFFFFFFFFu, b.rows[n], j);
      if (r < 0 || r >= s.rows_max) {                        // warp-uniform: not written
        if (lane == 0) raise_error(s.err, kErrBounds);
        continue;
      }
      if (active) {
        if (s.a_q != nullptr) *reinterpret_cast<uint4*>(s.a_q + r * (s.H / 2) + b.c0[n] / 2) = nib;
        if ((lane & 1) == 0) *reinterpret_cast<uint32_t*>(s.a_sf + sf_word_offset(r, k4, k4_total)) = word;
      }
    }
  }
}

// One warp stages all of token t (the side warps of the L2 GEMM): lane q < k
// holds slot q's row index (r_lane, loaded once per token by the caller), from
// which it forms the row's byte offsets in a_q and a_sf once; each segment
// takes them by shuffle.  The token's segments go in pairs, the loads of the
// next pair issued before the current pair is quantised and written.  A row
// outside [0, rows_max) is not written and sets kErrBounds.  (x_q is not
// written: the side job stages permuted rows only.)
__device__ __forceinline__ void stage_token_warp(const StageJob& s, int64_t t, int32_t r_lane, int lane) {
  const int segs = (s.H + 1023) / 1024;
  const int64_t k4_total = s.H / 64;
  const bool ok = lane < s.k && r_lane >= 0 && r_lane < s.rows_max;
  if (__any_sync(0xFFFFFFFFu, lane < s.k && !ok) && lane == 0) raise_error(s.err, kErrBounds);
  const int64_t q_off = ok ? static_cast<int64_t>(r_lane) * (s.H / 2) : -1;
  const int64_t sf_off = ok ? (static_cast<int64_t>(r_lane >> 7) * k4_total) * 512 + (r_lane & 31) * 16 +
                                  ((r_lane >> 5) & 3) * 4
                            : -1;
  const float g = s.x_gscale != nullptr ? __ldg(s.x_gscale) : 1.0f;
  const uint4* xrow = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(s.x) + t * s.H);
  auto load = [&](int seg, uint4 (&raw)[4]) {
    const int c0 = seg * 1024 + lane * 32;
    if (seg < segs && c0 < s.H) {
#pragma unroll
      for (int i = 0; i < 4; ++i) raw[i] = __ldg(xrow + c0 / 8 + i);
    }
  };
  auto store = [&](int seg, const uint4 (&raw)[4]) {
    if (seg >= segs) return;                   // warp-uniform
    const int c0 = seg * 1024 + lane * 32;
    const bool active = c0 < s.H;
    uint4 nib = make_uint4(0, 0, 0, 0);
    uint32_t codes = 0;
    if (active) stage_quantize(raw, s.x_gscale != nullptr, g, nib, codes);
    const uint32_t word = codes | (__shfl_down_sync(0xFFFFFFFFu, codes, 1) << 16);
    const int64_t sf_col = static_cast<int64_t>(c0 / 64) * 512;
    for (int j = 0; j < s.k; ++j) {
      const int64_t qo = __shfl_sync(0xFFFFFFFFu, q_off, j);
      const int64_t so = __shfl_sync(0xFFFFFFFFu, sf_off, j);
      if (qo < 0) continue;                    // warp-uniform: reported above
      if (active) {
        *reinterpret_cast<uint4*>(s.a_q + qo + c0 / 2) = nib;
        if ((lane & 1) == 0) *reinterpret_cast<uint32_t*>(s.a_sf + so + sf_col) = word;
      }
    }
  };
  uint4 ra[2][4], rb[2][4];
  load(0, ra[0]);
  load(1, ra[1]);
  for (int seg = 0; seg < segs; seg += 4) {
    load(seg + 2, rb[0]);
    load(seg + 3, rb[1]);
    store(seg, ra[0]);
    store(seg + 1, ra[1]);
    load(seg + 4, ra[0]);
    load(seg + 5, ra[1]);
    store(seg + 2, rb[0]);
    store(seg + 3, rb[1]);
  }
}

}  // namespace nvfp4

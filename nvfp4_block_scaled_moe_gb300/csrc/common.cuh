// Device helpers shared by the NVFP4 MoE kernels (sm_103a): NVFP4 numerics,
// bounded mbarrier waits, TMA / bulk copies and tcgen05 (TMEM, block-scaled MMA)
// wrappers written as inline PTX.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4 {

// ------------------------------------------------------------ error word --
// Bits of the per-device error word (a __device__ variable owned by abi.cu,
// passed to kernels as a pointer).
enum : unsigned { kErrTimeout = 1u, kErrBounds = 2u };

// A bounded wait gives up after this long; no legitimate wait in these kernels
// comes within orders of magnitude of it.
constexpr uint64_t kWaitLimitNs = 4000000000ull;

__device__ __forceinline__ void raise_error(unsigned* err, unsigned bits) {
  if (err != nullptr) atomicOr(err, bits);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// --------------------------------------------------------- NVFP4 numerics --
// E4M3 encode of a non-negative fp32 with round-to-nearest-even and saturation
// to 448 (cvt ... satfinite never produces the exp=15/mant=7 NaN for finite input).
__device__ __forceinline__ uint32_t e4m3_from_f32(float x) {
  uint16_t packed;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(packed) : "f"(0.0f), "f"(x));
  return packed & 0xFFu;   // the second source operand lands in the low byte
}

// Exact value of a non-negative E4M3 code (bias 7; e == 0 is m * 2^-9).
__device__ __forceinline__ float f32_from_e4m3(uint32_t code) {
  const uint32_t e = (code >> 3) & 0xFu, m = code & 7u;
  return e == 0 ? static_cast<float>(m) * 0.001953125f
                : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Pack eight half-step values (each a signed multiple of 0.5 in [-6, 6]) into
// eight E2M1 nibbles, element 2i in the low nibble of byte i.  Every input is
// already on the half-step grid, so the conversion's round-to-nearest-even only
// resolves the grid ties 2.5 -> 2, 3.5 -> 4, 5 -> 4 (ties to the even mantissa).
__device__ __forceinline__ uint32_t e2m1x8_from_halfsteps(const float (&v)[8]) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return out;
}

// RN(a / 6) for a >= 0 without a division routine.  y = RN(1/6) = 0x3E2AAAAB
// (1/6 = 1.0101...b x 2^-3; the 24th significant bit and a nonzero tail round the
// 23-bit fraction 0x2AAAAA up).  Markstein's theorem: with y = RN(1/b), q a
// faithful approximation of a/b and r = a - b*q (exact through the FMA),
// RN(q + r*y) = RN(a/b).  Results below 2^-126 may differ, which cannot change an
// E4M3 code (everything below 2^-10 encodes as 0).
__device__ __forceinline__ float div6_rn(float a) {
  const float y = __uint_as_float(0x3E2AAAABu);
  const float q0 = a * y;
  const float r = fmaf(-q0, 6.0f, a);
  return fmaf(r, y, q0);
}

// Block scale of a 16-block from its amax: E4M3(fp32(amax / 6)).  Kept as
// d2 = d/2 and r2 = RN(1/d2) = 2 RN(1/d) (exact scalings) so that the per-value
// path yields the half-step count 2|x|/d directly.
struct BlockScale {
  uint32_t code;  // E4M3 byte
  float d2;       // decoded scale / 2 (0 for a zero scale)
  float r2;       // RN(2 / decoded scale), 0 for a zero scale
};

__device__ __forceinline__ BlockScale block_scale(float amax) {
  BlockScale s;
  s.code = e4m3_from_f32(div6_rn(amax));
  s.d2 = 0.5f * f32_from_e4m3(s.code);
  s.r2 = s.d2 > 0.0f ? __frcp_rn(s.d2) : 0.0f;
  return s;
}

// Signed half step of x / d: rne(2 * x / d) / 2, which the E2M1 conversion then
// maps onto its grid (saturating above 6).
// q = RN(x / d2) = RN(2x / d) is the IEEE quotient, obtained from the correctly
// rounded reciprocal r2 with one FMA residual correction (Markstein, as in
// div6_rn).  The residual is taken as q0 * d2 - x and subtracted, which gives the
// same q and keeps the sign of a zero quotient (x = -0 or a zero scale -> -0).
// rintf (cvt.rni) rounds q to an integer with ties to even and keeps the sign, so
// a negative x whose magnitude rounds to 0 yields -0 (the E2M1 code 0x8).  For
// |q| <= 12 this equals copysign(rne(2 * min(|x / d|, 6)), x) / 2; above, both
// give a value >= 6 that the saturating conversion turns into the code of 6.
__device__ __forceinline__ float signed_halfstep(float x, const BlockScale& s) {
  const float q0 = x * s.r2;
  const float rem = fmaf(q0, s.d2, -x);
  const float q = fmaf(-rem, s.r2, q0);
  return rintf(q) * 0.5f;
}

// alpha of group g under the two-level encode scales of A (scalar) and B (per
// group): alpha / (ga * gb[g]) as one IEEE quotient; alpha itself when neither
// scale is given.
__device__ __forceinline__ float group_alpha(float alpha, const float* ga, const float* gb, int g) {
  if (ga == nullptr && gb == nullptr) return alpha;
  const float a = ga != nullptr ? __ldg(ga) : 1.0f;
  const float b = gb != nullptr ? __ldg(gb + g) : 1.0f;
  return __fdiv_rn(alpha, a * b);
}

// signed_halfstep of two values at once: the same IEEE round-to-nearest
// multiplies and FMAs, issued as packed two-lane fp32 instructions (sm_100 and
// later), so each lane's result is bit-identical to the scalar form.
__device__ __forceinline__ float2 signed_halfstep2(float2 x, const BlockScale& s) {
  const float2 r2 = make_float2(s.r2, s.r2);
  const float2 q0 = __fmul2_rn(x, r2);
  const float2 rem = __ffma2_rn(q0, make_float2(s.d2, s.d2), make_float2(-x.x, -x.y));
  const float2 q = __ffma2_rn(make_float2(-rem.x, -rem.y), r2, q0);
  return __fmul2_rn(make_float2(rintf(q.x), rintf(q.y)), make_float2(0.5f, 0.5f));
}

// Quantise eight values of one half-block with that block's scale.
__device__ __forceinline__ uint32_t quantize8(const float (&h)[8], const BlockScale& s) {
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const float2 t = signed_halfstep2(make_float2(h[i], h[i + 1]), s);
    v[i] = t.x;
    v[i + 1] = t.y;
  }
  return e2m1x8_from_halfsteps(v);
}

// silu(g) * u = g * u / (1 + 2^(-g * log2(e))), with the SFU's ex2.approx and
// rcp.approx (a few ulp; g -> -inf gives a signed zero, g -> +inf gives g * u).
__device__ __forceinline__ float swiglu(float g, float u) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(g * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return g * r * u;
}

// swiglu of two pairs: the same operations, the multiplies and the add issued
// as packed two-lane fp32 instructions (bit-identical per lane).
__device__ __forceinline__ float2 swiglu2(float2 g, float2 u) {
  const float2 t = __fmul2_rn(g, make_float2(-1.4426950408889634f, -1.4426950408889634f));
  float e0, e1, r0, r1;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(t.x));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(t.y));
  const float2 den = __fadd2_rn(make_float2(1.0f, 1.0f), make_float2(e0, e1));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(den.x));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(den.y));
  return __fmul2_rn(__fmul2_rn(g, make_float2(r0, r1)), u);
}

// Byte offset of the SF word holding scales (row, 4*k4 .. 4*k4+3) in the
// swizzled layout with k4_total 64-element column groups.
__device__ __forceinline__ uint64_t sf_word_offset(uint64_t row, uint32_t k4, uint32_t k4_total) {
  return ((row >> 7) * k4_total + k4) * 512ull + (row & 31u) * 16u + ((row >> 5) & 3u) * 4u;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& w, float (&f)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// The compact BF16 SwiGLU output of one thread's row: 128 interleaved gate/up
// accumulator columns (4 chunks of g(8) u(8) g(8) u(8)) -> 64 values of
// silu(alpha g) * (alpha u), rounded to BF16 and stored as 8 x 16 bytes at dst.
__device__ __forceinline__ void swiglu_bf16_row(const float (&v)[4][32], float alpha, __nv_bfloat16* dst) {
  uint4* out = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = 16 * half + 2 * i;
        w[i] = pack_bf16x2(swiglu(alpha * v[c][j], alpha * v[c][j + 8]),
                           swiglu(alpha * v[c][j + 1], alpha * v[c][j + 9]));
      }
      out[2 * c + half] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// One warp's share of the combine of token t (moe_combine's arithmetic: fp32
// FMA in slot order starting from 0, one rounding to BF16), in groups of
// 32 kNC 8-column chunks.  Lane q < k holds slot q's row index and weight
// (r_lane, w_lane, loaded once per token); every group takes them by shuffle,
// so no load waits on an index.  Pairs of values are accumulated with two-lane
// FMAs (each lane the same IEEE fmaf).  The rows are read once, with the
// evict-first hint (ld.global.cs): with plain loads the stream pushed the
// GEMM's reused operands out of L2 and the launch read 0.38 GB more from DRAM.
// A slot whose row lies outside [0, n_rows) loads nothing, adds 0 and sets
// kErrBounds.
template <int kNC>
__device__ __forceinline__ void combine_token_warp(const __nv_bfloat16* __restrict__ rows, int64_t n_rows,
                                                   int32_t r_lane, float w_lane, int32_t H, int32_t k, int64_t t,
                                                   __nv_bfloat16* __restrict__ y, int lane, unsigned* err) {
  constexpr int kGroup = 32 * kNC;
  const int chunks = H / 8;
  const int groups = (chunks + kGroup - 1) / kGroup;
  if (__any_sync(0xFFFFFFFFu, lane < k && (r_lane < 0 || r_lane >= n_rows)) && lane == 0)
    raise_error(err, kErrBounds);
  for (int g = 0; g < groups; ++g) {
    const int c0 = g * kGroup + lane;
    float2 acc[kNC][4];
#pragma unroll
    for (int n = 0; n < kNC; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[n][i] = make_float2(0.0f, 0.0f);
    for (int j0 = 0; j0 < k; j0 += 8) {
      uint4 v[8][kNC];
      float wj[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int j = j0 + q < k ? j0 + q : 0;                 // warp-uniform
        const int32_t r = __shfl_sync(0xFFFFFFFFu, r_lane, j);
        wj[q] = __shfl_sync(0xFFFFFFFFu, w_lane, j);
        const bool in = j0 + q < k && r >= 0 && r < n_rows;
        const uint4* src = reinterpret_cast<const uint4*>(rows + static_cast<int64_t>(in ? r : 0) * H);
#pragma unroll
        for (int n = 0; n < kNC; ++n)
          v[q][n] = in && c0 + 32 * n < chunks ? __ldcs(src + c0 + 32 * n) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (j0 + q < k) {
          const float2 w2 = make_float2(wj[q], wj[q]);
#pragma unroll
          for (int n = 0; n < kNC; ++n) {
            float f[8];
            bf16x8_to_f32(v[q][n], f);
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[n][i] = __ffma2_rn(w2, make_float2(f[2 * i], f[2 * i + 1]), acc[n][i]);
          }
        }
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(y + t * H);
#pragma unroll
    for (int n = 0; n < kNC; ++n)
      if (c0 + 32 * n < chunks)
        dst[c0 + 32 * n] = make_uint4(pack_bf16x2(acc[n][0].x, acc[n][0].y), pack_bf16x2(acc[n][1].x, acc[n][1].y),
                                      pack_bf16x2(acc[n][2].x, acc[n][2].y), pack_bf16x2(acc[n][3].x, acc[n][3].y));
  }
}

// --------------------------------------------------------- leftover blocks --
// The CTA-pair GEMM pairs consecutive 128-row blocks of a group, so a group with
// an odd block count ends in a pair tile whose odd CTA has no rows: the pair
// still stages and multiplies a whole tile for half of one.  With a split, a
// single-CTA launch on S SMs runs beside the pair launch of P clusters and takes
// the last block of some of those groups: the last n_take odd groups in group
// order (experts with few rows come last under a skewed routing, so the split
// takes the thin, weight-streaming ones first, whose DRAM time then overlaps the
// pair launch's compute-bound tiles instead of forming its tail), n_take chosen
// so that both launches end together.  A single-CTA 128-row tile costs its SM
// `cost` times what a full pair tile costs each of its two SMs, as it stages
// all 256 weight rows itself (54 instead of 38 KiB per K stage): measured best
// at 3/2 with a long K (at least kLeftLongK stages: the L1 GEMM) and 5/4 with a
// short one (the L2 GEMM, where the pair tile's accumulator hand-off weighs
// more).  So
//   n_take = min(n_odd, floor(S * (pairs + n_odd) / (P * cost + S))),
// pairs the full pairs over all groups.  Both kernels compute the same split
// from the offsets and K alone; S == 0: none.
constexpr int kLeftLongK = 16;                                  // K stages of 256
constexpr int64_t kLeftCostLongNum = 3, kLeftCostLongDen = 2;
constexpr int64_t kLeftCostShortNum = 5, kLeftCostShortDen = 4;
struct LeftoverSplit {
  int32_t n_odd;
  int32_t n_take;
};

// One warp, all lanes: the split over the G groups of the block offsets s_off.
__device__ __forceinline__ LeftoverSplit leftover_split(const int32_t* s_off, int G, int P, int S, int k_blocks,
                                                        int lane) {
  uint32_t pairs = 0, odd = 0;
  for (int g = lane; g < G; g += 32) {
    const int32_t blocks = (s_off[g + 1] - s_off[g]) / 128;
    if (blocks > 0) {
      pairs += static_cast<uint32_t>(blocks >> 1);
      odd += static_cast<uint32_t>(blocks & 1);
    }
  }
  pairs = __reduce_add_sync(0xFFFFFFFFu, pairs);
  odd = __reduce_add_sync(0xFFFFFFFFu, odd);
  LeftoverSplit ls;
  ls.n_odd = static_cast<int32_t>(odd);
  ls.n_take = 0;
  if (S > 0 && P > 0) {
    const bool long_k = k_blocks >= kLeftLongK;
    const int64_t num = long_k ? kLeftCostLongNum : kLeftCostShortNum;
    const int64_t den = long_k ? kLeftCostLongDen : kLeftCostShortDen;
    const int64_t fit = static_cast<int64_t>(S) * den * (static_cast<int64_t>(pairs) + odd) /
                        (static_cast<int64_t>(P) * num + static_cast<int64_t>(S) * den);
    ls.n_take = static_cast<int32_t>(fit < static_cast<int64_t>(odd) ? fit : static_cast<int64_t>(odd));
  }
  return ls;
}

// Inclusive warp scan of v (lane order).
__device__ __forceinline__ int32_t warp_scan_incl(int32_t v, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int32_t o = __shfl_up_sync(0xFFFFFFFFu, v, d);
    if (lane >= d) v += o;
  }
  return v;
}

// ------------------------------------------------------------- mbarriers --
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for the phase of `bar` with the given parity, but never forever: give up
// when *abort is set by another role, or after kWaitLimitNs (then set *abort and
// the timeout bit).  Returns true if the phase completed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                         unsigned* err, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort = 1;
        raise_error(err, kErrTimeout);
        return false;
      }
    }
  }
}

// All 32 lanes wait; the result is the same on every lane (false if any gave up).
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort,
                                              unsigned* err, uint64_t limit_ns = kWaitLimitNs) {
  const bool ok = mbar_wait(bar, parity, abort, err, limit_ns);
  return __all_sync(0xFFFFFFFFu, ok);
}

// ---------------------------------------------------------------- clusters --
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA in the cluster; release/acquire orders shared-memory
// writes (barrier initialisation included) before the other CTA's accesses.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in cluster CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(const void* p, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
  return out;
}

// One arrival on a barrier given by its shared::cluster address (possibly in the
// other CTA of the cluster).  Used to hand TMEM back after tcgen05.wait::ld and
// tcgen05.fence::before_thread_sync, which order the TMEM reads; the default
// (CTA-scope) release is enough for that and measurably cheaper than a
// cluster-scope release.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// One lane of a converged warp (the lowest active one) is elected.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// ----------------------------------------------------------- TMA / bulk --
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 2-D tiled load; x (innermost, in elements) must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// 2-D tiled load into this CTA's shared memory whose completion is counted on
// the barrier at cluster address `bar` (this CTA's or the other CTA's of the
// pair: the cta_group::2 form).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                                                 int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// Gather of four rows y.x .. y.w (each one 128-byte box row of a map whose box
// is 128 bytes x 1 row) into consecutive 128-byte rows at dst (which keeps the
// map's swizzle, as a 4-row tile at that address would); x as for tma_load_2d.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t x, int4 y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y.x), "r"(y.y), "r"(y.z), "r"(y.w)
      : "memory");
}

// The same, completing on the barrier at cluster address `bar` (cta_group::2).
__device__ __forceinline__ void tma_gather4_pair(void* dst, const CUtensorMap* map, uint32_t bar, int32_t x, int4 y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(bar), "r"(x), "r"(y.x), "r"(y.y), "r"(y.z), "r"(y.w)
      : "memory");
}

// Source rows of one 128-row block of A under a gather index: lane l gets the
// entries of rows 4l .. 4l+3.  Entries < 0 mark rows whose scales are zero
// (group padding) and read row 0; entries >= a_rows set the bounds bit and read
// row 0 too, so no copy leaves the matrix.
__device__ __forceinline__ int4 gather_rows4(const int32_t* index, int64_t block, int64_t a_rows, unsigned* err,
                                             int lane) {
  int4 r = __ldg(reinterpret_cast<const int4*>(index + block * 128) + lane);
  int* v = reinterpret_cast<int*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (v[i] >= a_rows) {
      raise_error(err, kErrBounds);
      v[i] = 0;
    }
    if (v[i] < 0) v[i] = 0;
  }
  return r;
}

// Contiguous global -> shared copy; both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tiled store from shared memory (bulk-group completion); x as for loads.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// This thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// This thread's committed bulk stores are complete (written to global memory).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Make this thread's generic-proxy shared-memory writes visible to TMA.
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05 --
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far completes.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Copy a 32-row x 16-byte shared-memory tile into TMEM, replicated to all four
// 32-lane groups (the scale-factor staging of the block-scaled MMA).
__device__ __forceinline__ void tc_copy_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// D(tmem) (+)= A(smem) * B(smem)^T, E2M1 x E2M1 with one UE4M3 scale per 16 K
// elements of A rows (sfa_tmem) and B rows (sfb_tmem); K = 64 per instruction.
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// --- CTA-pair forms (cta_group::2).  The two CTAs of a 2-CTA cluster share one
// MMA of M = 256: each supplies its 128 rows of A, its half of B's N rows and its
// own scale factors from its own shared memory, and holds its 128 accumulator
// rows in its own TMEM.  Allocation is collective (one warp in each CTA); MMAs,
// scale copies and commits are issued by the even CTA only.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Arrive once on `bar` (this CTA) when the pair operations issued so far complete.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// The same, arriving on the barrier at `bar`'s offset in every CTA of cta_mask.
__device__ __forceinline__ void tc_commit_pair_mc(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// Scale-factor atom copy into both CTAs' TMEM, each from its own shared memory.
__device__ __forceinline__ void tc_copy_sf_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void tc_mma_nvf4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Load 128 consecutive fp32 columns of this thread's TMEM lane (one instruction)
// and wait for them.
#define NVFP4_R32(o) "=r"(r[o + 0]), "=r"(r[o + 1]), "=r"(r[o + 2]), "=r"(r[o + 3]), "=r"(r[o + 4]), \
    "=r"(r[o + 5]), "=r"(r[o + 6]), "=r"(r[o + 7]), "=r"(r[o + 8]), "=r"(r[o + 9]), "=r"(r[o + 10]),        \
    "=r"(r[o + 11]), "=r"(r[o + 12]), "=r"(r[o + 13]), "=r"(r[o + 14]), "=r"(r[o + 15]), "=r"(r[o + 16]),   \
    "=r"(r[o + 17]), "=r"(r[o + 18]), "=r"(r[o + 19]), "=r"(r[o + 20]), "=r"(r[o + 21]), "=r"(r[o + 22]),   \
    "=r"(r[o + 23]), "=r"(r[o + 24]), "=r"(r[o + 25]), "=r"(r[o + 26]), "=r"(r[o + 27]), "=r"(r[o + 28]),   \
    "=r"(r[o + 29]), "=r"(r[o + 30]), "=r"(r[o + 31])
__device__ __forceinline__ void tmem_load128(uint32_t taddr, float (&v)[4][32]) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {"
      "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,"
      "%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,"
      "%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
      "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,"
      "%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,"
      "%126,%127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : NVFP4_R32(0), NVFP4_R32(32), NVFP4_R32(64), NVFP4_R32(96)
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i >> 5][i & 31] = __uint_as_float(r[i]);
}

#undef NVFP4_R32

// Load 32 consecutive fp32 columns of this thread's TMEM lane and wait for them.
__device__ __forceinline__ void tmem_load32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor (tcgen05 format, version 1) for a K-major
// operand tile written by TMA with 128-byte swizzle: 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;             // leading offset (unused with this swizzle)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;     // stride between 8-row groups
  d |= static_cast<uint64_t>(1u) << 46;             // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;             // 128-byte swizzle
  return d;
}

// Descriptor for a scale-factor atom: unswizzled 8 x 16-byte core matrices,
// consecutive along M|N, 128 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(128u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  return d;
}

// Instruction descriptor of kind::mxf4nvf4: E2M1 A and B (format code 1), both
// K-major, UE4M3 scales, scale-factor ids 0, dense K = 64.
__host__ __device__ constexpr uint32_t idesc_nvf4(uint32_t m, uint32_t n) {
  return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

}  // namespace nvfp4

// Block-scaled NVFP4 grouped GEMM on the sm_100-family tensor cores (tcgen05),
// with two fused epilogues:
//   * SwiGLU + NVFP4 re-quantisation (the L1 "fused_swiglu" kernel of "NVFP4-1.1
//     Approach, Part 2", in the fp4 mode the pages planned but could not build:
//     gate subtile -> SiLU in registers, up subtile -> SwiGLU, every 16 values ->
//     amax, E4M3 scale, E2M1 nibbles, written straight to global memory with the
//     scales in the swizzled MMA layout);
//   * alpha * acc -> BF16 rows (the L2 GEMM).
//
// Shape of the work: a tile is 128 rows x 256 columns of the output (one
// tcgen05.mma of M=128, N=256, K=64 per 64 K elements -- the N=256 shape keeps
// the tensor pipe busiest); the K loop runs in stages of 256 elements (128
// bytes of E2M1 per row = one 128-byte swizzle row).  Rows are grouped
// (experts): group g owns rows [offsets[g], offsets[g+1]) (multiples of 128)
// and multiplies with B_g.  As a split's single-CTA half (Params::left_ctas) the
// kernel computes only the last block of some odd groups, beside the CTA-pair
// kernel on the rest of the GPU (gemm_pair.cu; the rule is common.cuh's
// leftover_split).
//
// One persistent CTA per SM, 10 warps, warp-specialised:
//   warp 0     TMA producer: A (128 rows) and B (256 rows) tiles through 2-D tensor
//              maps with 128-byte swizzle, and the scale-factor atoms (contiguous
//              2 KiB bulk copies) into a 4-stage shared-memory ring;
//   warp 1     TMEM owner and MMA issuer: copies the stage's scale atoms into TMEM
//              (tcgen05.cp 32x128b.warpx4) and issues four tcgen05.mma kind::mxf4nvf4
//              block_scale scale_vec::4X per stage into the fp32 accumulator;
//   warps 2-9  epilogue, two warps per TMEM lane quadrant (one output row per
//              thread, 128 accumulator columns per warp).  Each warp copies its
//              columns from TMEM into registers and releases the accumulator at
//              once, so the next tile's MMAs run while it computes and stores.
// The producer and MMA warps run converged with warp-uniform operands and issue
// through one elected lane.  Lessons kept from the pages' pipeline notes: the
// first MMA of a tile does not accumulate; barrier arrival counts are in the
// units that actually arrive.  Every wait is bounded (a timeout sets the error
// word and lets the CTA exit).
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kBM = 128, kBK = 256;                    // elements
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kABytes = kBM * kBK / 2;            // 16 KiB
constexpr uint32_t kSfaBytes = kBM * (kBK / 16);       // 2 KiB: 4 atoms of 512 B
constexpr int kMaxGroups = 1024;
constexpr int kSplitCtas = 8;          // SMs of a split's single-CTA launch (four pair slots)
constexpr uint32_t kTmemCols = 512;

// Tile configuration by output-tile width BN:
//   BN = 256 (the L1 / SwiGLU kernel, long K): one 256-column accumulator, 4 stages;
//   BN = 128 (the BF16 kernel, L2's short K = I): two 128-column accumulators so
//     the next tile's MMAs overlap the hand-off of the previous one, 6 stages.
// TMEM: the accumulators first, then per stage 16 columns of A scales (4 atoms x
// 4 columns) and 16 per 128-row band of B scales.
template <int BN>
struct Cfg {
  static constexpr int kBN = BN;
  static constexpr int kAcc = BN == 256 ? 1 : 2;
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr int kBands = BN / 128;
  static constexpr int kChunks = BN / 64;              // 32-column chunks per epilogue warp
  static constexpr uint32_t kBBytes = BN * kBK / 2;
  static constexpr uint32_t kSfbBytes = BN * (kBK / 16);
  static constexpr uint32_t kStageTx = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr uint32_t kOffA = 0;
  static constexpr uint32_t kOffB = kOffA + kStages * kABytes;
  static constexpr uint32_t kOffSfa = kOffB + kStages * kBBytes;
  static constexpr uint32_t kOffSfb = kOffSfa + kStages * kSfaBytes;
  static constexpr uint32_t kOffBar = kOffSfb + kStages * kSfbBytes;
  static constexpr uint32_t kNumBars = 2 * kStages + 2 * kAcc + 1;   // full, empty, tfull, tempty, drain
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;     // tmem slot, abort flag
  static constexpr uint32_t kOffGroups = kOffMisc + 16;
  static constexpr uint32_t kOffLeft = kOffGroups + (kMaxGroups + 1) * 4;  // a split's leftover blocks, count
  static constexpr uint32_t kSmemBytes = kOffLeft + (kPairMaxGroups + 1) * 4 + 1024;   // + alignment slack
  static constexpr uint32_t kTmemSf = kAcc * BN;
  static constexpr uint32_t kTmemSfStage = 16 + 16 * kBands;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffB % 1024 == 0 && kOffSfa % 1024 == 0, "swizzled tiles need 1 KiB alignment");
  static_assert(kTmemSf + kStages * kTmemSfStage <= kTmemCols, "TMEM budget");
};

struct Params {
  const uint8_t* a_sf;
  const uint8_t* b_sf;
  const int32_t* a_gather;    // null, or the source row in A of every padded row
  int64_t a_rows;
  const int32_t* offsets;
  const int32_t* counts;
  int32_t G, N, K;
  int32_t n_tiles, k_blocks;
  int64_t rows_max;
  int64_t sfb_group_bytes;
  float alpha;
  const float* a_gs;          // two-level encode scales (null = 1): A, B per group, SwiGLU output
  const float* b_gs;
  const float* out_gs;
  uint8_t* out_q;
  uint8_t* out_sf;
  __nv_bfloat16* out_bf16;
  float* h_debug;
  unsigned* err;
  // left_ctas > 0: this launch is a split's single-CTA half (common.cuh:
  // leftover_split, beside a pair launch of pair_clusters clusters) and computes
  // only the last block of the odd groups it takes, thinnest groups first
  int32_t left_ctas, pair_clusters;
};

__device__ __forceinline__ int find_group(const int32_t* off, int G, int64_t row) {
  int lo = 0, hi = G;                 // last g < G with off[g] <= row
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= row) lo = mid; else hi = mid;
  }
  return lo;
}

// L1 epilogue for one thread's row: 128 interleaved gate/up accumulator columns
// (4 chunks of g(8) u(8) g(8) u(8)) -> 64 SwiGLU outputs -> 4 NVFP4 blocks (of
// fp32(h * g_out) under a two-level encode scale; h_debug keeps h).
__device__ __forceinline__ void epilogue_swiglu(const float (&v)[4][32], float alpha, const float* out_gs,
                                                bool valid, int64_t grow, int64_t col0, int32_t out_cols,
                                                uint32_t k4, uint32_t k4_total, uint8_t* out_q, uint8_t* out_sf,
                                                float* h_debug) {
  uint32_t sf_word = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float h0[8], h1[8];
    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      const float2 t0 = swiglu2(__fmul2_rn(a2, make_float2(v[c][i], v[c][i + 1])),
                                __fmul2_rn(a2, make_float2(v[c][8 + i], v[c][9 + i])));
      const float2 t1 = swiglu2(__fmul2_rn(a2, make_float2(v[c][16 + i], v[c][17 + i])),
                                __fmul2_rn(a2, make_float2(v[c][24 + i], v[c][25 + i])));
      h0[i] = t0.x;
      h0[i + 1] = t0.y;
      h1[i] = t1.x;
      h1[i + 1] = t1.y;
    }
    const int64_t col = col0 + 16 * c;
    if (valid && h_debug != nullptr) {
      float4* hp = reinterpret_cast<float4*>(h_debug + grow * out_cols + col);
      hp[0] = make_float4(h0[0], h0[1], h0[2], h0[3]);
      hp[1] = make_float4(h0[4], h0[5], h0[6], h0[7]);
      hp[2] = make_float4(h1[0], h1[1], h1[2], h1[3]);
      hp[3] = make_float4(h1[4], h1[5], h1[6], h1[7]);
    }
    if (out_gs != nullptr) {
      const float g = __ldg(out_gs);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        h0[i] *= g;
        h1[i] *= g;
      }
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fmaxf(fabsf(h0[i]), fabsf(h1[i])));
    const BlockScale s = block_scale(amax);
    const uint32_t lo = quantize8(h0, s), hi = quantize8(h1, s);
    sf_word |= s.code << (8 * c);
    if (valid) *reinterpret_cast<uint2*>(out_q + grow * (out_cols / 2) + col / 2) = make_uint2(lo, hi);
  }
  if (valid) *reinterpret_cast<uint32_t*>(out_sf + sf_word_offset(grow, k4, k4_total)) = sf_word;
}

// L2 epilogue for one thread's row: alpha * (32 * kChunks) accumulator columns -> BF16.
template <int kChunks>
__device__ __forceinline__ void epilogue_bf16(const float (&v)[kChunks][32], float alpha, __nv_bfloat16* dst_row) {
  uint4* dst = reinterpret_cast<uint4*>(dst_row);
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 o;
      o.x = pack_bf16x2(alpha * v[c][8 * q + 0], alpha * v[c][8 * q + 1]);
      o.y = pack_bf16x2(alpha * v[c][8 * q + 2], alpha * v[c][8 * q + 3]);
      o.z = pack_bf16x2(alpha * v[c][8 * q + 4], alpha * v[c][8 * q + 5]);
      o.w = pack_bf16x2(alpha * v[c][8 * q + 6], alpha * v[c][8 * q + 7]);
      dst[4 * c + q] = o;
    }
  }
}

// kGather: A rows come through p.a_gather (tile::gather4); a separate
// instantiation, so the default kernels carry none of its code.
template <int kEpi, int BN, bool kGather>
__global__ void __launch_bounds__(kThreads, 1)
    nvf4_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                     const Params p) {
  using C = Cfg<BN>;
  constexpr int kStages = C::kStages, kAcc = C::kAcc, kBN = C::kBN, kBands = C::kBands;
  constexpr uint32_t kBBytes = C::kBBytes, kSfbBytes = C::kSfbBytes, kStageTx = C::kStageTx;
  constexpr uint32_t kOffA = C::kOffA, kOffB = C::kOffB, kOffSfa = C::kOffSfa, kOffSfb = C::kOffSfb;
  constexpr uint32_t kTmemSf = C::kTmemSf, kTmemSfStage = C::kTmemSfStage;
  static_assert(kEpi == NVFP4_EPI_BF16 || BN == 256, "the SwiGLU epilogues use 256-column tiles");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + kAcc;
  uint64_t* drain = tempty + kAcc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + C::kOffGroups);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < kAcc; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiWarps);    // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i <= p.G; i += blockDim.x)
    s_off[i] = p.offsets != nullptr ? __ldg(p.offsets + i) : (i == 0 ? 0 : static_cast<int32_t>(p.rows_max));
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmap_a);
    tma_prefetch_map(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  // a split's leftover blocks: s_left[i] is the last block of the i-th group
  // taken, counting from the last odd group down; s_left[kPairMaxGroups] the count
  int32_t* s_left = reinterpret_cast<int32_t*>(smem + C::kOffLeft);
  if (p.left_ctas > 0) {
    if (warp == 2) {
      const LeftoverSplit ls = leftover_split(s_off, p.G, p.pair_clusters, p.left_ctas, p.k_blocks, lane);
      int32_t carry_odd = 0;
      for (int base = 0; base < p.G; base += 32) {
        const int g = base + lane;
        int32_t blocks = 0;
        if (g < p.G) blocks = (s_off[g + 1] - s_off[g]) / kBM;
        if (blocks < 0) blocks = 0;
        const int32_t odd = blocks & 1;
        const int32_t rank = carry_odd + warp_scan_incl(odd, lane) - odd;     // odd groups before g
        const int32_t from_last = ls.n_odd - 1 - rank;
        if (odd != 0 && from_last < ls.n_take && from_last < kPairMaxGroups)
          s_left[from_last] = s_off[g + 1] / kBM - 1;
        carry_odd += __reduce_add_sync(0xFFFFFFFFu, static_cast<uint32_t>(odd));
      }
      if (lane == 0) s_left[kPairMaxGroups] = ls.n_take < kPairMaxGroups ? ls.n_take : kPairMaxGroups;
    }
    __syncthreads();
  }

  // the grouped rows must be a 128-aligned prefix of the allocation
  const int64_t total_rows = s_off[p.G];
  int64_t num_tiles = 0;
  if (total_rows >= 0 && total_rows <= p.rows_max && (total_rows % kBM) == 0) {
    num_tiles = (p.left_ctas > 0 ? s_left[kPairMaxGroups] : total_rows / kBM) * p.n_tiles;
  } else if (threadIdx.x == 0) {
    raise_error(p.err, kErrBounds);
  }
  const int32_t k4 = p.K / 64;        // scale atoms per 128-row band

  // The producer and MMA warps run their loops with all 32 lanes converged, so
  // every descriptor, coordinate and TMEM address is warp-uniform (held in the
  // uniform datapath); one elected lane issues the TMA / tcgen05 instructions.
  const uint32_t tmem_u = __shfl_sync(0xFFFFFFFFu, tmem_base, 0);
  const int64_t tiles_u = __shfl_sync(0xFFFFFFFFu, num_tiles, 0);
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t stage = 0, phase = 0, filled = 0, fill_parity = 0;
    bool ok = true;
    for (int64_t tile = blockIdx.x; tile < tiles_u && ok; tile += gridDim.x) {
      const int64_t mi = tile / p.n_tiles;
      const int32_t nt = static_cast<int32_t>(tile - mi * p.n_tiles);
      const int64_t mt = p.left_ctas > 0 ? s_left[mi] : mi;
      const int g = __shfl_sync(0xFFFFFFFFu, find_group(s_off, p.G, mt * kBM), 0);
      const uint8_t* sfa = p.a_sf + (mt * k4) * 512;
      const uint8_t* sfb = p.b_sf + g * p.sfb_group_bytes + (static_cast<int64_t>(kBands * nt) * k4) * 512;
      constexpr bool gather = kGather;
      const int4 rows4 = gather ? gather_rows4(p.a_gather, mt, p.a_rows, p.err, lane) : make_int4(0, 0, 0, 0);
      for (int32_t kb = 0; kb < p.k_blocks; ++kb) {
        ok = mbar_wait_warp(&empty[stage], phase ^ 1u, abort_flag, p.err);
        if (!ok) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&full[stage], kStageTx);
          if (!gather)
            tma_load_2d(smem + kOffA + stage * kABytes, &tmap_a, &full[stage], kb * (kBK / 2),
                        static_cast<int32_t>(mt * kBM));
          tma_load_2d(smem + kOffB + stage * kBBytes, &tmap_b, &full[stage], kb * (kBK / 2), g * p.N + nt * kBN);
          bulk_load(smem + kOffSfa + stage * kSfaBytes, sfa + kb * 4 * 512, kSfaBytes, &full[stage]);
#pragma unroll
          for (int b = 0; b < kBands; ++b)     // one 2 KiB run of 4 atoms per 128-row band of B
            bulk_load(smem + kOffSfb + stage * kSfbBytes + b * 2048, sfb + (b * k4 + kb * 4) * 512, 2048,
                      &full[stage]);
        }
        __syncwarp();
        // gathered A: every lane copies its 4 rows (the byte count is in the expect_tx above)
        if constexpr (gather) {
          tma_gather4(smem + kOffA + stage * kABytes + lane * 512, &tmap_a, &full[stage], kb * (kBK / 2), rows4);
          __syncwarp();
        }
        filled |= 1u << stage;
        fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) {
      // let the copies already in flight land before the CTA can exit
      int no_abort = 0;
      for (int s = 0; s < kStages; ++s)
        if ((filled >> s) & 1u) mbar_wait(&full[s], (fill_parity >> s) & 1u, &no_abort, nullptr, 50000000ull);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = idesc_nvf4(kBM, kBN);
    uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
    bool ok = true;
    for (int64_t tile = blockIdx.x; tile < tiles_u && ok; tile += gridDim.x) {
      ok = mbar_wait_warp(&tempty[acc], acc_phase ^ 1u, abort_flag, p.err);
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t d_tmem = tmem_u + acc * kBN;
      for (int32_t kb = 0; kb < p.k_blocks; ++kb) {
        ok = mbar_wait_warp(&full[stage], phase, abort_flag, p.err);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t sfa_t = tmem_u + kTmemSf + stage * kTmemSfStage;
        const uint32_t sfb_t = sfa_t + 16;
        const uint32_t sfa_s = smem_u32(smem + kOffSfa + stage * kSfaBytes);
        const uint32_t sfb_s = smem_u32(smem + kOffSfb + stage * kSfbBytes);
        const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(smem + kOffA + stage * kABytes));
        const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(smem + kOffB + stage * kBBytes));
        if (elect_one()) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            tc_copy_sf(sfa_t + 4 * j, sdesc_sf(sfa_s + 512 * j));
#pragma unroll
            for (int b = 0; b < kBands; ++b)   // B rows 128b .. 128b+127
              tc_copy_sf(sfb_t + 4 * kBands * j + 4 * b, sdesc_sf(sfb_s + 2048 * b + 512 * j));
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // K advance of 64 E2M1 = 32 bytes inside the 128-byte swizzle row
            tc_mma_nvf4(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sfa_t + 4 * j, sfb_t + 4 * kBands * j,
                        (kb | j) != 0 ? 1u : 0u);
          }
          tc_commit(&empty[stage]);
        }
        __syncwarp();
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (elect_one()) tc_commit(&tfull[acc]);
      __syncwarp();
      if (++acc == kAcc) { acc = 0; acc_phase ^= 1u; }
    }
    // every MMA issued by the elected lane has completed before the CTA moves on
    if (elect_one()) tc_commit(drain);
    __syncwarp();
    int no_abort = 0;
    mbar_wait(drain, 0, &no_abort, p.err, 100000000ull);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const uint32_t quad = warp & 3;                // TMEM lanes 32*quad .. +31
    const uint32_t half = (warp - 2) >> 2;         // accumulator columns (kBN/2)*half .. +kBN/2-1
    const uint32_t row_in_tile = quad * 32 + lane;
    uint32_t acc = 0, acc_phase = 0;
    for (int64_t tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const int64_t mi = tile / p.n_tiles;
      const int32_t nt = static_cast<int32_t>(tile - mi * p.n_tiles);
      const int64_t mt = p.left_ctas > 0 ? s_left[mi] : mi;
      const int64_t grow = mt * kBM + row_in_tile;
      const int g = find_group(s_off, p.G, mt * kBM);
      bool valid = true;
      if (p.counts != nullptr) valid = (grow - s_off[g]) < __ldg(p.counts + g);
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, p.err)) break;
      tc_fence_after_sync();
      float v[C::kChunks][32];
      const uint32_t t_row = tmem_base + ((quad * 32u) << 16) + acc * kBN + half * (kBN / 2);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) tmem_load32(t_row + 32 * c, v[c]);
      // the accumulator is in registers: hand it back to the MMA warp
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == kAcc) { acc = 0; acc_phase ^= 1u; }
      const float alpha = group_alpha(p.alpha, p.a_gs, p.b_gs, g);
      if constexpr (kEpi == NVFP4_EPI_SWIGLU_NVFP4) {
        epilogue_swiglu(v, alpha, p.out_gs, valid, grow, static_cast<int64_t>(nt) * (kBN / 2) + half * 64, p.N / 2,
                        2 * nt + half, static_cast<uint32_t>(p.N / 128), p.out_q, p.out_sf, p.h_debug);
      } else if constexpr (kEpi == NVFP4_EPI_SWIGLU_BF16) {
        if (valid)
          swiglu_bf16_row(v, alpha, p.out_bf16 + grow * (p.N / 2) + static_cast<int64_t>(nt) * (kBN / 2) + half * 64);
      } else {
        if (valid)
          epilogue_bf16<C::kChunks>(v, alpha,
                                    p.out_bf16 + grow * p.N + static_cast<int64_t>(nt) * kBN + half * (kBN / 2));
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ host --
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

}  // namespace

// rows x cols matrix of elem_bytes-sized elements (row-major, rows contiguous),
// box of box_cols x box_rows, optionally with 128-byte swizzle.
bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t rows, uint64_t cols,
                  uint32_t elem_bytes, uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * elem_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

std::atomic<int> g_gemm_tiles{NVFP4_GEMM_TILES_AUTO};

struct DeviceInfo {
  int sms = 0;
  bool attr_set[5] = {false, false, false, false, false};
};

DeviceInfo& device_info(int dev) {
  static DeviceInfo info[64];
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& d = info[dev & 63];
  if (d.sms == 0) cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  return d;
}

// The stream a split's single-CTA launch runs on, one per device (created on
// first use, never destroyed; the caller's stream forks to it and joins it back
// through events, so calls on any streams and under capture stay ordered).
cudaStream_t split_stream(int dev) {
  static cudaStream_t streams[64] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  cudaStream_t& s = streams[dev & 63];
  if (s == nullptr && cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) s = nullptr;
  return s;
}

// A split's single-CTA half: 128-row tiles over the leftover blocks, on `ctas`
// CTAs launched as clusters of two, so that they take whole pair slots and the
// pair launch beside them keeps all of its clusters resident.
template <int kEpi>
cudaError_t launch_left(const CUtensorMap& ma, const CUtensorMap& mb, const Params& p, int ctas, cudaStream_t stream,
                        DeviceInfo& info) {
  constexpr int slot = kEpi == NVFP4_EPI_SWIGLU_NVFP4 ? 0 : kEpi == NVFP4_EPI_SWIGLU_BF16 ? 3 : 1;
  if (!info.attr_set[slot]) {
    cudaError_t e = cudaFuncSetAttribute(nvf4_gemm_kernel<kEpi, 256, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg<256>::kSmemBytes));
    if (e != cudaSuccess) return e;
    info.attr_set[slot] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg<256>::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, nvf4_gemm_kernel<kEpi, 256, false>, ma, mb, p);
}

template <int kEpi, int BN, bool kGather = false>
cudaError_t launch(const CUtensorMap& ma, const CUtensorMap& mb, const Params& p, int grid, cudaStream_t stream,
                   DeviceInfo& info) {
  constexpr int slot = kGather ? 4
                       : kEpi == NVFP4_EPI_SWIGLU_NVFP4 ? 0 : kEpi == NVFP4_EPI_SWIGLU_BF16 ? 3 : (BN == 256 ? 1 : 2);
  if (!info.attr_set[slot]) {
    cudaError_t e = cudaFuncSetAttribute(nvf4_gemm_kernel<kEpi, BN, kGather>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg<BN>::kSmemBytes));
    if (e != cudaSuccess) return e;
    info.attr_set[slot] = true;
  }
  nvf4_gemm_kernel<kEpi, BN, kGather><<<grid, kThreads, Cfg<BN>::kSmemBytes, stream>>>(ma, mb, p);
  return cudaGetLastError();
}

}  // namespace

nvfp4_status gemm_launch(const GemmArgs& a, cudaStream_t stream) {
  if (a.G > kMaxGroups) return fail(NVFP4_ERR_UNSUPPORTED, "nvfp4_grouped_gemm: G=%d exceeds %d", a.G, kMaxGroups);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  DeviceInfo& info = device_info(dev);
  if (info.sms <= 0) return fail(NVFP4_ERR_CUDA, "nvfp4_grouped_gemm: no SM count for device %d", dev);

  // 128x256 tiles whenever N allows (an N=256 MMA does twice an N=128 MMA's work
  // for about 1.4x its issue cost, which outweighs the single-buffered
  // accumulator's hand-off); BF16 outputs with N an odd multiple of 128 use
  // 128x128 tiles with a double-buffered accumulator.  Groups averaging two or
  // more 128-row blocks go to the CTA-pair kernel (256x256 tiles, gemm_pair.cu);
  // thinner groups (decode-sized batches) would leave half of many pair tiles empty.
  const bool swiglu = a.epilogue != NVFP4_EPI_BF16;
  const int bn = (swiglu || a.N % 256 == 0) ? 256 : 128;
  const int mode = g_gemm_tiles.load(std::memory_order_relaxed);
  const int64_t groups = a.offsets != nullptr ? a.G : 1;
  const bool pair = bn == 256 && groups <= kPairMaxGroups &&
                    (mode == NVFP4_GEMM_TILES_PAIR ||
                     (mode == NVFP4_GEMM_TILES_AUTO && a.rows_max >= 2 * kBM * groups));
  // side jobs: the combine of an earlier batch runs inside the CTA-pair SwiGLU
  // kernel, the activation staging of a later batch inside the CTA-pair BF16
  // kernel; a job the chosen kernel does not host runs as its own launch first,
  // and so does one whose GEMM has tiles for fewer than half the SMs (the side
  // warps would then be too few to stream it)
  const int64_t pair_tiles = ((a.rows_max / kBM + 1) / 2 + (groups > 1 ? groups : 0)) * (a.N / 256);
  const bool wide = pair_tiles * 2 >= info.sms / 2;
  const bool host_combine = pair && wide && a.epilogue == NVFP4_EPI_SWIGLU_NVFP4 && a.a_gather == nullptr;
  const bool host_stage = pair && wide && a.epilogue == NVFP4_EPI_BF16 && a.a_gather == nullptr;
  if ((a.side_T > 0 && !host_combine) || (a.stage.T > 0 && !host_stage)) {
    GemmArgs rest = a;
    if (a.side_T > 0 && !host_combine) {
      e = combine_launch(a.side_rows, a.side_n_rows, a.side_inv, a.side_w, a.side_T, a.side_H, a.side_k, nullptr,
                         a.side_y, stream);
      if (e != cudaSuccess) return fail_cuda(e, "nvfp4_grouped_gemm: combine of the earlier batch");
      rest.side_T = 0;
    }
    if (a.stage.T > 0 && !host_stage) {
      e = stage_launch(a.stage, stream);
      if (e != cudaSuccess) return fail_cuda(e, "nvfp4_grouped_gemm: staging of the later batch");
      rest.stage.T = 0;
    }
    return gemm_launch(rest, stream);
  }
  // a grouped CTA-pair GEMM (auto tiles) is split: kSplitCtas SMs run a
  // single-CTA launch over the last block of the thinnest odd groups beside
  // the pair launch, which skips those groups' half-empty pair tiles
  const bool split = pair && mode == NVFP4_GEMM_TILES_AUTO && a.offsets != nullptr && a.G > 1 &&
                     a.a_gather == nullptr && info.sms >= 8 * kSplitCtas;
  if (pair && !split) return gemm_pair_launch(a, info.sms, dev, stream);
  CUtensorMap ma, mb;
  const bool gather = a.a_gather != nullptr;      // gathered A rows: a one-row box for tile::gather4
  if (!make_tmap_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.a_q,
                    static_cast<uint64_t>(gather ? a.a_rows : a.rows_max), static_cast<uint64_t>(a.K) / 2, 1, 128,
                    gather ? 1 : kBM, true) ||
      !make_tmap_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.b_q, static_cast<uint64_t>(a.G) * a.N,
                    static_cast<uint64_t>(a.K) / 2, 1, 128, bn, true))
    return fail(NVFP4_ERR_CUDA, "nvfp4_grouped_gemm: cuTensorMapEncodeTiled failed");

  Params p;
  p.a_sf = a.a_sf;
  p.b_sf = a.b_sf;
  p.a_gather = a.a_gather;
  p.a_rows = a.a_rows;
  p.offsets = a.offsets;
  p.counts = a.counts;
  p.G = a.offsets != nullptr ? a.G : 1;
  p.N = a.N;
  p.K = a.K;
  p.n_tiles = a.N / bn;
  p.k_blocks = a.K / kBK;
  p.rows_max = a.rows_max;
  p.sfb_group_bytes = static_cast<int64_t>(a.N / 128) * (a.K / 64) * 512;
  p.alpha = a.alpha;
  p.a_gs = a.a_gscale;
  p.b_gs = a.b_gscale;
  p.out_gs = a.out_gscale;
  p.out_q = a.out_q;
  p.out_sf = a.out_sf;
  p.out_bf16 = static_cast<__nv_bfloat16*>(a.out_bf16);
  p.h_debug = a.h_debug;
  p.err = device_error_word();
  p.left_ctas = 0;
  p.pair_clusters = 0;

  if (split) {
    cudaStream_t side = split_stream(dev);
    if (side == nullptr) return fail(NVFP4_ERR_CUDA, "nvfp4_grouped_gemm: no split stream");
    cudaEvent_t fork = nullptr, join = nullptr;
    e = cudaEventCreateWithFlags(&fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&join, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(fork, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side, fork, 0);
    nvfp4_status st = NVFP4_OK;
    int clusters = 0;
    if (e == cudaSuccess) st = gemm_pair_launch(a, info.sms, dev, stream, kSplitCtas, &clusters);
    if (e == cudaSuccess && st == NVFP4_OK) {
      p.left_ctas = kSplitCtas;
      p.pair_clusters = clusters;
      e = a.epilogue == NVFP4_EPI_SWIGLU_NVFP4 ? launch_left<NVFP4_EPI_SWIGLU_NVFP4>(ma, mb, p, kSplitCtas, side, info)
          : a.epilogue == NVFP4_EPI_SWIGLU_BF16 ? launch_left<NVFP4_EPI_SWIGLU_BF16>(ma, mb, p, kSplitCtas, side, info)
                                                : launch_left<NVFP4_EPI_BF16>(ma, mb, p, kSplitCtas, side, info);
      if (e == cudaSuccess) e = cudaEventRecord(join, side);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, join, 0);
    }
    if (fork != nullptr) cudaEventDestroy(fork);
    if (join != nullptr) cudaEventDestroy(join);
    if (st != NVFP4_OK) return st;
    if (e != cudaSuccess) return fail_cuda(e, "nvfp4_grouped_gemm: split launch");
    return NVFP4_OK;
  }

  const int64_t max_tiles = (a.rows_max / kBM) * p.n_tiles;
  const int grid = static_cast<int>(max_tiles < info.sms ? max_tiles : info.sms);
  if (grid <= 0) return NVFP4_OK;
  e = gather                                ? launch<NVFP4_EPI_SWIGLU_NVFP4, 256, true>(ma, mb, p, grid, stream, info)
      : a.epilogue == NVFP4_EPI_SWIGLU_NVFP4 ? launch<NVFP4_EPI_SWIGLU_NVFP4, 256>(ma, mb, p, grid, stream, info)
      : a.epilogue == NVFP4_EPI_SWIGLU_BF16 ? launch<NVFP4_EPI_SWIGLU_BF16, 256>(ma, mb, p, grid, stream, info)
      : bn == 256                           ? launch<NVFP4_EPI_BF16, 256>(ma, mb, p, grid, stream, info)
                                            : launch<NVFP4_EPI_BF16, 128>(ma, mb, p, grid, stream, info);
  if (e != cudaSuccess) return fail_cuda(e, "nvfp4_grouped_gemm launch");
  return NVFP4_OK;
}

nvfp4_status set_gemm_tiles(int mode) {
  if (mode != NVFP4_GEMM_TILES_AUTO && mode != NVFP4_GEMM_TILES_SINGLE && mode != NVFP4_GEMM_TILES_PAIR)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_set_gemm_tiles: unknown mode %d", mode);
  g_gemm_tiles.store(mode, std::memory_order_relaxed);
  return NVFP4_OK;
}

}  // namespace nvfp4

// Block-scaled NVFP4 grouped GEMM on CTA pairs (tcgen05 cta_group::2): the
// same contraction and epilogues as gemm.cu's single-CTA kernel, for groups
// with enough rows to fill 256-row tiles.
//
// A 2-CTA cluster owns an output tile of 256 rows x 256 columns.  One
// tcgen05.mma of M=256, N=256, K=64 per 64 K elements, issued by the even CTA,
// multiplies both CTAs' 128 rows of A with the 256 rows of B, each CTA holding
// half of B in its own shared memory.  Per output element each SM therefore
// loads a third fewer operand bytes than a 128 x 256 single-CTA tile (A 16 KiB
// + half of B 16 KiB per 256-element K stage instead of 16 + 32 KiB), which
// lets the ring hold the same stage count in less shared memory.
//
// Rows are grouped (experts) as in gemm.cu: group g owns the 128-row blocks
// [offsets[g]/128, offsets[g+1]/128).  Tiles pair consecutive blocks of one
// group; a group with an odd block count ends in a tile whose odd CTA has no
// rows (it loads no A, computes a discarded half and stores nothing), unless a
// split's single-CTA launch beside this one takes that group's last block
// (PairParams::left_ctas; common.cuh: leftover_split), in which case the tile
// is skipped.
//
// Roles (320 threads per CTA, 384 with a side job; one CTA per SM):
//   warp 0     producer: TMA loads of A (128 rows), this CTA's 128 rows of B,
//              this CTA's A scale atoms and both 128-row bands of B's scale
//              atoms (every CTA multiplies against all 256 B rows, so each needs
//              both bands in its own TMEM).  Both CTAs' loads complete on the
//              even CTA's full barrier, which expects the pair's bytes
//              (cta_group::2 TMA);
//   warp 1     even CTA: TMEM owner and MMA issuer (scale copies and MMAs for
//              the pair, commits multicast to both CTAs' barriers); idle on the
//              odd CTA after the collective TMEM allocation;
//   warps 2-9  epilogue on this CTA's 128 accumulator rows, as in gemm.cu,
//              except that complete 32-row slices leave through shared memory:
//              BF16 rows are staged 64 columns at a time and written back with
//              each store instruction covering four whole 128-byte lines (instead
//              of 32 partial lines), the stores spaced out over the next tile's
//              mainloop; SwiGLU nibble rows leave by TMA store;
//   warps 10-11  (side-job instantiations only) an HBM-bound job of another
//              batch: the combine of an earlier batch beside the SwiGLU GEMM,
//              the activation staging of a later batch beside the BF16 GEMM.
// Every wait is bounded; a timeout sets the error word and the pair drains
// and exits together (the final cluster barrier keeps each CTA's shared
// memory alive while the other may still address it).
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "stage.cuh"

namespace nvfp4 {
namespace {

constexpr int kBM = 128, kBK = 256;                    // rows per CTA, K per stage
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kSideWarps = 2;                          // the side job's warps (kSide instantiations)
constexpr int kSideNone = 0, kSideCombine = 1, kSideStage = 2;
constexpr int kThreadsSide = kThreads + 32 * kSideWarps;
constexpr int kMaxGroups = kPairMaxGroups;             // larger G uses the single-CTA kernel
constexpr uint32_t kABytes = kBM * kBK / 2;            // 16 KiB
constexpr uint32_t kSfaBytes = kBM * (kBK / 16);       // 2 KiB: 4 atoms
constexpr uint32_t kTmemCols = 512;

// A pair tile is 256 rows x 256 columns, with one accumulator of 256 TMEM
// columns per CTA: a second does not fit beside the scale factors, so the MMAs
// of the next tile wait for the epilogue to drain it.  (Tiles of 256 x 128 with
// two accumulators would hide that wait but halve the operand reuse per byte
// staged in shared memory, whose bandwidth bounds this kernel; they measured
// slower on every shape.)
//
// Per epilogue: the staging buffer of one warp's output slice.
//   SwiGLU: 32 rows x 32 bytes of nibbles (one 1 KiB TMA-store box per tile);
//   BF16:   32 rows x 64 columns (4 KiB, 16-byte chunks XOR-swizzled by row).
template <int kEpi>
struct PairCfg {
  static constexpr bool kSwiglu = kEpi == NVFP4_EPI_SWIGLU_NVFP4;
  static constexpr int kBN = 256;                                    // columns of a pair tile
  static constexpr int kAcc = 1;                                     // accumulators in TMEM
  static constexpr int kBands = kBN / 128;                           // 128-row bands of B's scale atoms
  static constexpr int kChunks = kBN / 64;                           // 32-column chunks per epilogue warp
  static constexpr uint32_t kBBytes = (kBN / 2) * kBK / 2;           // this CTA's half of the B rows
  static constexpr uint32_t kSfbBytes = kBN * (kBK / 16);            // scale atoms of every B row
  static constexpr uint32_t kTmemSf = kAcc * kBN;                    // scale columns follow the accumulator
  static constexpr uint32_t kTmemSfStage = 16 + 16 * kBands;         // A: 4 atoms x 4 columns; B: 4 per band
  static constexpr int kStages = 5;
  static constexpr uint32_t kStageBufBytes = kSwiglu ? 1024 : 4096;
  static constexpr uint32_t kOffA = 0;
  static constexpr uint32_t kOffB = kOffA + kStages * kABytes;
  static constexpr uint32_t kOffSfa = kOffB + kStages * kBBytes;
  static constexpr uint32_t kOffSfb = kOffSfa + kStages * kSfaBytes;
  static constexpr uint32_t kOffOut = kOffSfb + kStages * kSfbBytes;
  static constexpr uint32_t kOffBar = kOffOut + kEpiWarps * kStageBufBytes;
  static constexpr uint32_t kNumBars = 2 * kStages + 2 * kAcc + 1;         // full, empty, tfull, tempty, drain
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;             // tmem slot, abort flag
  static constexpr uint32_t kOffGroups = kOffMisc + 16;                    // row offsets, then pair prefix
  static constexpr uint32_t kSmemBytes = kOffGroups + 2 * (kMaxGroups + 1) * 4;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffB % 1024 == 0 && kOffSfa % 1024 == 0 && kOffOut % 1024 == 0, "1 KiB alignment");
  static_assert(kTmemSf + kStages * kTmemSfStage <= kTmemCols, "TMEM budget");
};

struct PairParams {
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
  // side jobs, run by the two side warps of every CTA while the GEMM runs:
  // kSideCombine, the combine of an earlier batch (side_T == 0: none);
  // kSideStage, the activation staging of a later batch
  const __nv_bfloat16* side_rows;
  int64_t side_n_rows;
  const int32_t* side_inv;
  const float* side_w;
  __nv_bfloat16* side_y;
  int32_t side_T, side_H, side_k;
  StageJob stage;
  // split: a single-CTA launch of left_ctas CTAs runs beside this one (of
  // pair_clusters clusters) and takes the last block of some odd groups, whose
  // half-empty pair tiles this launch then skips (common.cuh: leftover_split);
  // left_ctas == 0: no split
  int32_t left_ctas, pair_clusters;
};

// last g < G with tab[g] <= v (tab non-decreasing, tab[0] = 0 <= v)
__device__ __forceinline__ int last_le(const int32_t* tab, int G, int64_t v) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tab[mid] <= v) lo = mid; else hi = mid;
  }
  return lo;
}

// Where a tile's rows live for CTA `rank` of the pair: tile = pair index (the
// group's consecutive 128-row block pairs) * n_tiles + 256-column tile.
struct TileRows {
  int g;            // group
  int32_t nt;       // the 256-column tile
  int64_t block;    // this CTA's 128-row block
  bool has_rows;    // the block belongs to group g (and to the allocation)
};

__device__ __forceinline__ TileRows tile_rows(const int32_t* s_off, const int32_t* s_pair, const PairParams& p,
                                              int64_t tile, uint32_t rank) {
  TileRows t;
  const int64_t pair = tile / p.n_tiles;
  t.nt = static_cast<int32_t>(tile - pair * p.n_tiles);
  t.g = last_le(s_pair, p.G, pair);
  t.block = s_off[t.g] / kBM + 2 * (pair - s_pair[t.g]) + rank;
  t.has_rows = t.block < s_off[t.g + 1] / kBM && t.block < p.rows_max / kBM;
  return t;
}

// SwiGLU + NVFP4 for one thread's row (128 interleaved accumulator columns ->
// 64 outputs -> 4 blocks): the 32 nibble bytes go to `stage` (or straight to
// global memory when `direct`), the scale word and h_debug straight to global.
__device__ __forceinline__ void swiglu_row(const float (&v)[4][32], float alpha, bool valid, bool direct,
                                           int64_t grow, int64_t col0, int32_t out_cols, uint32_t k4,
                                           uint32_t k4_total, uint8_t* stage_row, const PairParams& p) {
  uint32_t w[8];
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
    if (valid && p.h_debug != nullptr) {
      float4* hp = reinterpret_cast<float4*>(p.h_debug + grow * out_cols + col0 + 16 * c);
      hp[0] = make_float4(h0[0], h0[1], h0[2], h0[3]);
      hp[1] = make_float4(h0[4], h0[5], h0[6], h0[7]);
      hp[2] = make_float4(h1[0], h1[1], h1[2], h1[3]);
      hp[3] = make_float4(h1[4], h1[5], h1[6], h1[7]);
    }
    if (p.out_gs != nullptr) {                // two-level scale: quantise fp32(h * g)
      const float g = __ldg(p.out_gs);
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
    w[2 * c] = quantize8(h0, s);
    w[2 * c + 1] = quantize8(h1, s);
    sf_word |= s.code << (8 * c);
  }
  if (direct) {
    if (valid) {
      uint4* dst = reinterpret_cast<uint4*>(p.out_q + grow * (out_cols / 2) + col0 / 2);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  } else {
    uint4* dst = reinterpret_cast<uint4*>(stage_row);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
  if (valid) *reinterpret_cast<uint32_t*>(p.out_sf + sf_word_offset(grow, k4, k4_total)) = sf_word;
}

// Scale-factor atoms are loaded through 2-D maps of 256-byte rows: one 2 KiB
// run of four atoms is a box of 8 rows.
constexpr int kSfRow = 256;

// Returns once the SM clock reaches `due` (a fixed time: the wait ends).
__device__ __forceinline__ void wait_until_clock(long long due) {
  while (clock64() < due) __nanosleep(32);
}

// kGather: A rows come through p.a_gather (tile::gather4); a separate
// instantiation, so the default kernels carry none of its code.
// kSide: two more warps per CTA run an HBM-bound side job while the producer,
// MMA and epilogue warps run the GEMM, whose own DRAM traffic leaves room for
// it: the combine of an earlier batch (kSideCombine, in the SwiGLU L1 kernel)
// or the activation staging of a later batch (kSideStage, in the BF16 L2
// kernel).  Tokens are dealt to the side warps of all CTAs in turn, a warp
// taking a whole token.
template <int kEpi, bool kGather, int kSide>
__global__ void __launch_bounds__(kSide != kSideNone ? kThreadsSide : kThreads, 1)
    nvf4_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                          const __grid_constant__ CUtensorMap tmap_sfa, const __grid_constant__ CUtensorMap tmap_sfb,
                          const __grid_constant__ CUtensorMap tmap_out, const PairParams p) {
  using C = PairCfg<kEpi>;
  constexpr int kStages = C::kStages, kAcc = C::kAcc, kBN = C::kBN, kBands = C::kBands;
  constexpr uint32_t kBBytes = C::kBBytes, kSfbBytes = C::kSfbBytes;
  constexpr uint32_t kTmemSf = C::kTmemSf, kTmemSfStage = C::kTmemSfStage;
  extern __shared__ __align__(1024) uint8_t smem[];
  // the swizzled tiles need a 1 KiB-aligned base; every CTA sees the same base,
  // so a misaligned one stops all of them here, before any pair traffic
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) raise_error(p.err, kErrBounds);
    return;
  }
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + kAcc;
  uint64_t* drain = tempty + kAcc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + C::kOffGroups);
  int32_t* s_pair = s_off + (kMaxGroups + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();         // 0: the even CTA (MMA issuer), 1: the odd CTA
  const bool leader = rank == 0;
  const int64_t cluster_id = blockIdx.x / 2, n_clusters = gridDim.x / 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);                // the even CTA's: expect_tx of the pair's bytes
      mbar_init(&empty[s], 1);               // the pair's MMA commit (multicast to both CTAs)
    }
    for (int a = 0; a < kAcc; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * kEpiWarps);    // every epilogue warp of both CTAs (used on the even CTA)
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
    tma_prefetch_map(&tmap_sfa);
    tma_prefetch_map(&tmap_sfb);
    tma_prefetch_map(&tmap_out);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  __syncthreads();
  if (warp == 2) {
    // pair prefix: s_pair[g] = sum over groups before g of ceil(blocks / 2),
    // less the half-empty pair of each odd group a split's single-CTA launch takes
    const LeftoverSplit ls = leftover_split(s_off, p.G, p.pair_clusters, p.left_ctas, p.k_blocks, lane);
    int32_t carry = 0, carry_odd = 0;
    if (lane == 0) s_pair[0] = 0;
    for (int base = 0; base < p.G; base += 32) {
      const int g = base + lane;
      int32_t blocks = 0;
      if (g < p.G) blocks = (s_off[g + 1] - s_off[g]) / kBM;
      if (blocks < 0) blocks = 0;
      const int32_t odd = blocks & 1;
      const int32_t odd_incl = warp_scan_incl(odd, lane);
      const bool taken = odd != 0 && carry_odd + odd_incl - odd >= ls.n_odd - ls.n_take;
      const int32_t v = warp_scan_incl((blocks >> 1) + (odd != 0 && !taken ? 1 : 0), lane);
      if (g < p.G) s_pair[g + 1] = carry + v;
      carry += __shfl_sync(0xFFFFFFFFu, v, 31);
      carry_odd += __shfl_sync(0xFFFFFFFFu, odd_incl, 31);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();          // both CTAs' barriers and TMEM exist before any cross-CTA traffic
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  const int64_t total_rows = s_off[p.G];
  int64_t num_tiles = 0;
  if (total_rows >= 0 && total_rows <= p.rows_max && (total_rows % kBM) == 0) {
    num_tiles = static_cast<int64_t>(s_pair[p.G]) * p.n_tiles;
  } else if (threadIdx.x == 0) {
    raise_error(p.err, kErrBounds);
  }
  const int32_t k4 = p.K / 64;
  const uint32_t tmem_u = __shfl_sync(0xFFFFFFFFu, tmem_base, 0);
  const int64_t tiles_u = __shfl_sync(0xFFFFFFFFu, num_tiles, 0);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t stage = 0, phase = 0, filled = 0, fill_parity = 0;
    const uint32_t leader_full = mapa_shared(full, 0);
    bool ok = true;
    for (int64_t tile = cluster_id; tile < tiles_u && ok; tile += n_clusters) {
      const TileRows t = tile_rows(s_off, s_pair, p, tile, rank);
      const TileRows odd = tile_rows(s_off, s_pair, p, tile, 1);
      const int g = __shfl_sync(0xFFFFFFFFu, t.g, 0);
      const int64_t block = __shfl_sync(0xFFFFFFFFu, t.block, 0);
      const bool has_rows = __shfl_sync(0xFFFFFFFFu, t.has_rows, 0);
      const bool odd_rows = __shfl_sync(0xFFFFFFFFu, odd.has_rows, 0);
      // SF rows (256 bytes) of this block's A atoms and of the tile's two B bands
      const int32_t sfa_row = static_cast<int32_t>(block * k4 * (512 / kSfRow));
      const int64_t sfb_base = g * p.sfb_group_bytes + static_cast<int64_t>(kBands * t.nt) * k4 * 512;
      // the even CTA always has rows; both CTAs load B and its scales
      const uint32_t tx = 2 * (kBBytes + kSfbBytes) + (kABytes + kSfaBytes) + (odd_rows ? kABytes + kSfaBytes : 0u);
      constexpr bool gather = kGather;
      const int4 rows4 = gather && has_rows ? gather_rows4(p.a_gather, block, p.a_rows, p.err, lane)
                                            : make_int4(0, 0, 0, 0);
      for (int32_t kb = 0; kb < p.k_blocks; ++kb) {
        ok = mbar_wait_warp(&empty[stage], phase ^ 1u, abort_flag, p.err);
        if (!ok) break;
        const uint32_t bar = leader_full + 8u * stage;
        if (elect_one()) {
          if (leader) mbar_arrive_expect_tx(&full[stage], tx);
          if (has_rows) {
            if (!gather)
              tma_load_2d_pair(smem + C::kOffA + stage * kABytes, &tmap_a, bar, kb * (kBK / 2),
                               static_cast<int32_t>(block * kBM));
            tma_load_2d_pair(smem + C::kOffSfa + stage * kSfaBytes, &tmap_sfa, bar, 0, sfa_row + kb * 8);
          }
          tma_load_2d_pair(smem + C::kOffB + stage * kBBytes, &tmap_b, bar, kb * (kBK / 2),
                           g * p.N + t.nt * kBN + static_cast<int32_t>(rank) * (kBN / 2));
          // B's scale atoms: both bands (one 2 KiB run of four atoms each) into this CTA
#pragma unroll
          for (int b = 0; b < kBands; ++b) {
            const int64_t sfb_src = (static_cast<int64_t>(b) * k4 + kb * 4) * 512;
            tma_load_2d_pair(smem + C::kOffSfb + stage * kSfbBytes + b * 2048, &tmap_sfb, bar, 0,
                             static_cast<int32_t>((sfb_base + sfb_src) / kSfRow));
          }
        }
        __syncwarp();
        // gathered A: every lane copies its 4 rows (the bytes are in the pair's expect_tx)
        if (kGather && has_rows) {
          tma_gather4_pair(smem + C::kOffA + stage * kABytes + lane * 512, &tmap_a, bar, kb * (kBK / 2), rows4);
          __syncwarp();
        }
        filled |= 1u << stage;
        fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) {
      // let the copies already in flight land before the CTA can exit: the even
      // CTA waits on its barriers (which count the pair's bytes), the odd CTA
      // waits a fixed 1 ms
      int no_abort = 0;
      if (leader) {
        for (int s = 0; s < kStages; ++s)
          if ((filled >> s) & 1u) mbar_wait(&full[s], (fill_parity >> s) & 1u, &no_abort, nullptr, 50000000ull);
      } else {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) __nanosleep(1000);
      }
    }
    __syncwarp();
  } else if (warp == 1 && leader) {
    // ---------------------------------------------------- MMA issuer (pair)
    constexpr uint32_t idesc = idesc_nvf4(2 * kBM, kBN);
    uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
    bool ok = true;
    for (int64_t tile = cluster_id; tile < tiles_u && ok; tile += n_clusters) {
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
        const uint32_t sfa_s = smem_u32(smem + C::kOffSfa + stage * kSfaBytes);
        const uint32_t sfb_s = smem_u32(smem + C::kOffSfb + stage * kSfbBytes);
        const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(smem + C::kOffA + stage * kABytes));
        const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(smem + C::kOffB + stage * kBBytes));
        if (elect_one()) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            tc_copy_sf_pair(sfa_t + 4 * j, sdesc_sf(sfa_s + 512 * j));
#pragma unroll
            for (int b = 0; b < kBands; ++b)
              tc_copy_sf_pair(sfb_t + 4 * kBands * j + 4 * b, sdesc_sf(sfb_s + 2048 * b + 512 * j));
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc_mma_nvf4_pair(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sfa_t + 4 * j, sfb_t + 4 * kBands * j,
                             (kb | j) != 0 ? 1u : 0u);
          tc_commit_pair_mc(&empty[stage], 0x3);
        }
        __syncwarp();
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (elect_one()) tc_commit_pair_mc(&tfull[acc], 0x3);
      __syncwarp();
      if (++acc == kAcc) { acc = 0; acc_phase ^= 1u; }
    }
    if (elect_one()) tc_commit_pair(drain);
    __syncwarp();
    int no_abort = 0;
    mbar_wait(drain, 0, &no_abort, p.err, 100000000ull);
    __syncwarp();
  } else if (warp == 1) {
    // odd CTA: nothing to issue (the even CTA's MMAs read this CTA's stages)
  } else if (kSide != kSideNone && warp >= 2 + kEpiWarps) {
    // ----------------------------------------------------------- side job
    const int64_t sw = static_cast<int64_t>(blockIdx.x) * kSideWarps + (warp - 2 - kEpiWarps);
    const int64_t n_sw = static_cast<int64_t>(gridDim.x) * kSideWarps;
    if constexpr (kSide == kSideCombine) {
      // tokens dealt to the side warps in turn; lane q < k loads slot q's row
      // and weight of its warp's next token while the current one is combined
      auto slot = [&](int64_t t, int32_t& r, float& w) {
        r = -1;
        w = 0.0f;
        if (t < p.side_T && lane < p.side_k) {
          r = __ldg(p.side_inv + t * p.side_k + lane);
          w = __ldg(p.side_w + t * p.side_k + lane);
        }
      };
      int32_t r_cur, r_nxt;
      float w_cur, w_nxt;
      slot(sw, r_cur, w_cur);
      for (int64_t t = sw; t < p.side_T; t += n_sw) {
        slot(t + n_sw, r_nxt, w_nxt);
        combine_token_warp<3>(p.side_rows, p.side_n_rows, r_cur, w_cur, p.side_H, p.side_k, t, p.side_y, lane,
                              p.err);
        r_cur = r_nxt;
        w_cur = w_nxt;
      }
    } else {
      // the padding scales of expert e (one warp per expert), then the tokens,
      // dealt to the side warps in turn; lane q < k loads slot q's row of the
      // warp's next token while the current one is staged
      for (int e = static_cast<int>(sw); e < p.stage.E; e += static_cast<int>(n_sw)) stage_padding(p.stage, e, lane, 32);
      auto row = [&](int64_t t) {
        return t < p.stage.T && lane < p.stage.k ? __ldg(p.stage.inv_perm + t * p.stage.k + lane) : -1;
      };
      int32_t r_cur = row(sw);
      for (int64_t t = sw; t < p.stage.T; t += n_sw) {
        const int32_t r_nxt = row(t + n_sw);
        stage_token_warp(p.stage, t, r_cur, lane);
        r_cur = r_nxt;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const uint32_t quad = warp & 3;                // TMEM lanes 32*quad .. +31
    const uint32_t half = (warp - 2) >> 2;         // accumulator columns (kBN/2)*half .. +kBN/2-1
    const uint32_t row_in_tile = quad * 32 + lane;
    const uint32_t leader_tempty = mapa_shared(tempty, 0);
    uint8_t* stage_buf = smem + C::kOffOut + (warp - 2) * C::kStageBufBytes;
    uint32_t acc = 0, acc_phase = 0;
    bool stores_pending = false;
    // BF16 rows: each warp's 16 store instructions per tile (512 bytes each) are
    // spread over about 1.25 times the tile's MMA time at the instruction
    // ceiling (128 cycles per MMA, 4 MMAs per K stage), at most 320 cycles
    // apart.  Issued back to back by all eight warps they measured 6-8% slower
    // at K = 2048: the burst holds up the TMA loads of the next tile's stages.
    const long long store_gap = min(static_cast<long long>(p.k_blocks) * 40, 320LL);
    for (int64_t tile = cluster_id; tile < num_tiles; tile += n_clusters) {
      const TileRows t = tile_rows(s_off, s_pair, p, tile, rank);
      const int64_t grow = t.block * kBM + row_in_tile;
      bool valid = t.has_rows;
      if (valid && p.counts != nullptr) valid = (grow - s_off[t.g]) < __ldg(p.counts + t.g);
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, p.err)) break;
      tc_fence_after_sync();
      float v[C::kChunks][32];
      const uint32_t t_row = tmem_base + ((quad * 32u) << 16) + acc * kBN + half * (kBN / 2);
      tmem_load128(t_row, v);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(leader_tempty + 8u * acc);
      if (++acc == kAcc) { acc = 0; acc_phase ^= 1u; }

      // whole 32-row slices leave by TMA store; a slice with missing rows stores row by row
      const float alpha = group_alpha(p.alpha, p.a_gs, p.b_gs, t.g);
      const bool staged = __all_sync(0xFFFFFFFFu, valid);
      if (C::kSwiglu && staged) {
        if (lane == 0 && stores_pending) bulk_wait_read_all();
        __syncwarp();
      }
      const int32_t y = static_cast<int32_t>(t.block * kBM + quad * 32);
      if constexpr (C::kSwiglu) {
        swiglu_row(v, alpha, valid, !staged, grow, static_cast<int64_t>(t.nt) * (kBN / 2) + half * 64, p.N / 2,
                   2 * t.nt + half, static_cast<uint32_t>(p.N / 128), stage_buf + lane * 32, p);
        if (staged) {
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmap_out, stage_buf, t.nt * (kBN / 4) + half * 32, y);
            bulk_commit_group();
          }
          stores_pending = true;
        }
      } else if constexpr (kEpi == NVFP4_EPI_SWIGLU_BF16) {
        if (valid)
          swiglu_bf16_row(v, alpha, p.out_bf16 + grow * (p.N / 2) + static_cast<int64_t>(t.nt) * (kBN / 2) + half * 64);
      } else {
        if (staged) {
          // passes of 32 rows x 64 columns through the staging buffer: each
          // thread writes its row's 8 chunks of 16 bytes (chunk q of row r at
          // slot q ^ (r & 7), so 8 consecutive rows cover all banks), then each
          // store instruction takes 4 rows x 8 chunks = four whole 128-byte lines
          const int sub = lane >> 3, chunk = lane & 7;
          const long long t0 = clock64();
          const int64_t x = static_cast<int64_t>(t.nt) * kBN + half * (kBN / 2);
          uint8_t* my_row = stage_buf + lane * 128;
#pragma unroll
          for (int box = 0; box < C::kChunks / 2; ++box) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float* f = &v[2 * box + (q >> 2)][8 * (q & 3)];
              uint4 o;
              o.x = pack_bf16x2(alpha * f[0], alpha * f[1]);
              o.y = pack_bf16x2(alpha * f[2], alpha * f[3]);
              o.z = pack_bf16x2(alpha * f[4], alpha * f[5]);
              o.w = pack_bf16x2(alpha * f[6], alpha * f[7]);
              *reinterpret_cast<uint4*>(my_row + ((q ^ (lane & 7)) << 4)) = o;
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int row = 4 * i + sub;
              wait_until_clock(t0 + (box * 8 + i) * store_gap);
              const uint4 val =
                  *reinterpret_cast<const uint4*>(stage_buf + row * 128 + ((chunk ^ (row & 7)) << 4));
              // streaming store: the rows are read back only by the combine, from HBM
              __stcs(reinterpret_cast<uint4*>(p.out_bf16 + (static_cast<int64_t>(y) + row) * p.N + x + box * 64 +
                                              chunk * 8),
                     val);
            }
            __syncwarp();
          }
        } else if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(p.out_bf16 + grow * p.N + static_cast<int64_t>(t.nt) * kBN +
                                                half * (kBN / 2));
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c) {
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
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();          // neither CTA frees TMEM or exits while the pair may still touch it
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

struct PairDeviceInfo {
  bool attr_set[6] = {};
  int max_clusters[6] = {};
};

PairDeviceInfo& pair_info(int dev) {
  static PairDeviceInfo info[64];
  return info[dev & 63];
}

std::mutex& pair_mutex() {
  static std::mutex mu;
  return mu;
}

// reserve: clusters' worth of SMs left free for a split's single-CTA launch (the
// launch's cluster count goes to p.pair_clusters and *clusters_out)
template <int kEpi, bool kGather, int kSide = kSideNone>
cudaError_t launch_pair(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& msa, const CUtensorMap& msb,
                        const CUtensorMap& mo, PairParams p, int64_t num_tiles, int sms, int dev,
                        cudaStream_t stream, int reserve, int* clusters_out) {
  constexpr int slot = kSide != kSideNone ? 3 + kSide
                       : kGather          ? 3
                                          : (kEpi == NVFP4_EPI_SWIGLU_NVFP4 ? 0 : kEpi == NVFP4_EPI_BF16 ? 1 : 2);
  constexpr uint32_t smem = PairCfg<kEpi>::kSmemBytes;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kSide != kSideNone ? kThreadsSide : kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int max_clusters = 0;
  {
    std::lock_guard<std::mutex> lock(pair_mutex());
    PairDeviceInfo& info = pair_info(dev);
    if (!info.attr_set[slot]) {
      cudaError_t e = cudaFuncSetAttribute(nvf4_gemm_pair_kernel<kEpi, kGather, kSide>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      cfg.gridDim = dim3(static_cast<unsigned>(sms / 2 * 2), 1, 1);
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, nvf4_gemm_pair_kernel<kEpi, kGather, kSide>, &cfg);
      if (e != cudaSuccess) return e;
      info.max_clusters[slot] = n;
      info.attr_set[slot] = true;
    }
    max_clusters = info.max_clusters[slot];
  }
  // every cluster resident at once (the tile loop strides by the cluster count)
  const int64_t avail = static_cast<int64_t>(max_clusters) - reserve;
  int64_t clusters = avail < num_tiles ? avail : num_tiles;
  if (clusters <= 0) return cudaErrorInvalidConfiguration;
  p.pair_clusters = static_cast<int32_t>(clusters);
  if (clusters_out != nullptr) *clusters_out = static_cast<int>(clusters);
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
  return cudaLaunchKernelEx(&cfg, nvf4_gemm_pair_kernel<kEpi, kGather, kSide>, ma, mb, msa, msb, mo, p);
}

}  // namespace

nvfp4_status gemm_pair_launch(const GemmArgs& a, int sms, int dev, cudaStream_t stream, int left_ctas,
                              int* clusters_out) {
  if (a.G > kMaxGroups) return fail(NVFP4_ERR_UNSUPPORTED, "nvfp4_grouped_gemm: G=%d exceeds %d", a.G, kMaxGroups);
  constexpr int bn = PairCfg<NVFP4_EPI_BF16>::kBN;      // pair tile columns
  const bool swiglu = a.epilogue == NVFP4_EPI_SWIGLU_NVFP4;
  CUtensorMap ma, mb, msa, msb, mo;
  const uint64_t sfa_bytes = static_cast<uint64_t>(a.rows_max / 128) * (a.K / 64) * 512;
  const uint64_t sfb_bytes = static_cast<uint64_t>(a.G) * (a.N / 128) * (a.K / 64) * 512;
  const bool gather = a.a_gather != nullptr;      // gathered A rows: a one-row box for tile::gather4
  bool ok = make_tmap_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.a_q,
                         static_cast<uint64_t>(gather ? a.a_rows : a.rows_max), static_cast<uint64_t>(a.K) / 2, 1,
                         128, gather ? 1 : 128, true) &&
            make_tmap_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.b_q, static_cast<uint64_t>(a.G) * a.N,
                         static_cast<uint64_t>(a.K) / 2, 1, 128, static_cast<uint32_t>(bn / 2), true) &&
            make_tmap_2d(&msa, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.a_sf, sfa_bytes / kSfRow, kSfRow, 1, kSfRow, 8,
                         false) &&
            make_tmap_2d(&msb, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.b_sf, sfb_bytes / kSfRow, kSfRow, 1, kSfRow, 8,
                         false);      // one 128-row band's four atoms per box
  if (swiglu)
    ok = ok && make_tmap_2d(&mo, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.out_q, static_cast<uint64_t>(a.rows_max),
                            static_cast<uint64_t>(a.N) / 4, 1, 32, 32, false);
  else   // BF16 outputs: [rows_max, N], or [rows_max, N/2] for the compact SwiGLU output
    ok = ok && make_tmap_2d(&mo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.out_bf16, static_cast<uint64_t>(a.rows_max),
                            static_cast<uint64_t>(a.epilogue == NVFP4_EPI_BF16 ? a.N : a.N / 2), 2, 64, 32, true);
  if (!ok) return fail(NVFP4_ERR_CUDA, "nvfp4_grouped_gemm: cuTensorMapEncodeTiled failed");

  PairParams p;
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
  const bool side = a.side_T > 0;
  const bool stage = a.stage.T > 0;
  p.side_rows = static_cast<const __nv_bfloat16*>(a.side_rows);
  p.side_n_rows = a.side_n_rows;
  p.side_inv = a.side_inv;
  p.side_w = a.side_w;
  p.side_y = static_cast<__nv_bfloat16*>(a.side_y);
  p.side_T = a.side_T;
  p.side_H = a.side_H;
  p.side_k = a.side_k;
  p.stage = a.stage;
  p.left_ctas = left_ctas;
  p.pair_clusters = 0;

  // tiles that can exist: every group's pairs, at most ceil(blocks / 2) + G
  const int64_t blocks = a.rows_max / kBM;
  const int64_t max_pairs = (blocks + 1) / 2 + (p.G > 1 ? p.G : 0);
  const int64_t max_tiles = max_pairs * p.n_tiles;
  if (max_tiles <= 0) return NVFP4_OK;
  const int reserve = (left_ctas + 1) / 2;
#define NVFP4_PAIR_LAUNCH(E, GA) \
  launch_pair<E, GA>(ma, mb, msa, msb, mo, p, max_tiles, sms, dev, stream, reserve, clusters_out)
  const cudaError_t e = side ? launch_pair<NVFP4_EPI_SWIGLU_NVFP4, false, kSideCombine>(
                                   ma, mb, msa, msb, mo, p, max_tiles, sms, dev, stream, reserve, clusters_out)
                        : stage ? launch_pair<NVFP4_EPI_BF16, false, kSideStage>(
                                      ma, mb, msa, msb, mo, p, max_tiles, sms, dev, stream, reserve, clusters_out)
                        : gather                              ? NVFP4_PAIR_LAUNCH(NVFP4_EPI_SWIGLU_NVFP4, true)
                        : swiglu                              ? NVFP4_PAIR_LAUNCH(NVFP4_EPI_SWIGLU_NVFP4, false)
                        : a.epilogue == NVFP4_EPI_SWIGLU_BF16 ? NVFP4_PAIR_LAUNCH(NVFP4_EPI_SWIGLU_BF16, false)
                                                              : NVFP4_PAIR_LAUNCH(NVFP4_EPI_BF16, false);
#undef NVFP4_PAIR_LAUNCH
  if (e != cudaSuccess) return fail_cuda(e, "nvfp4_grouped_gemm (CTA pairs) launch");
  return NVFP4_OK;
}

}  // namespace nvfp4

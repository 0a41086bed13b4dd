// Routing, padded expert permutation, activation staging and the weighted combine.
//
// "NVFP4 MegaMoE Debug Log", section "NVFP4 MoE Pipeline": stage_activation of
// the hidden states, and the final scatter with routing weights.  "NVFP4-1.1
// Approach, Part 2": the padded per-expert layout (padded_dst gather / scatter).
//
// The permutation is deterministic although it counts with atomics: tokens are
// cut into chunks of kRouteChunk; the top-k kernel counts each chunk's rows per
// expert (shared-memory atomic increments commute), one block turns the chunk
// counts into per-chunk bases and the 128-padded expert offsets, and each chunk
// then ranks its rows of every expert by token order (bit masks of the tokens
// that picked it).  Rows of an expert therefore come in ascending token order.
// The activation staging (stage.cuh) follows as its own launch, or runs later
// on the side warps of an L2 GEMM.
#include <float.h>

#include "common.cuh"
#include "internal.h"
#include "stage.cuh"

namespace nvfp4 {

size_t route_workspace_bytes(int32_t T, int32_t E) {
  const size_t n_chunks = (static_cast<size_t>(T) + kRouteChunk - 1) / kRouteChunk;
  return ((n_chunks * static_cast<size_t>(E) * sizeof(int32_t) + 255) & ~static_cast<size_t>(255)) + 256;
}

void route_carve_workspace(RouteBuffers& b, void* workspace) {
  b.chunk_hist = static_cast<int32_t*>(workspace);
}

// Order-preserving 64-bit key of (logit, expert): larger logit first, and among
// equal logits the lower expert index first (-0.0 and +0.0 compare equal).
__device__ __forceinline__ uint64_t topk_key(float v, int e) {
  const uint32_t bits = __float_as_uint(v + 0.0f);
  const uint32_t ord = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
  return (static_cast<uint64_t>(ord) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(e));
}

__device__ __forceinline__ float key_value(uint64_t key) {
  const uint32_t ord = static_cast<uint32_t>(key >> 32);
  return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}

// ------------------------------------------------------------------ top-k --
// One block per chunk of kRouteChunk tokens, one warp per token at a time: each
// lane holds the logits of experts lane + 32j (j < kKeys, kKeys = ceil(E / 32))
// as order-preserving 32-bit codes, and its best remaining one (the lowest j
// among equal codes).  Each of the k rounds takes the warp's largest code with
// one redux.sync max, then the lowest expert holding it with one redux.sync min:
// larger logit first, lower expert index among equal logits.
// The chunk's per-expert counts gather in shared memory and leave as one row of
// the chunk histogram (no global atomics, nothing to clear beforehand).  Short
// batches (few chunks) split each chunk over gridDim.y blocks, so that every
// warp ranks one token; those blocks add their counts into the cleared row.
constexpr int kTopkThreads = 1024;

// This lane's logits of token t as codes; 0 sorts below every finite logit
// (absent experts, and later the taken ones).
template <int kKeys>
__device__ __forceinline__ void topk_load(const float* __restrict__ logits, int64_t t, int32_t E, int lane,
                                          uint32_t (&code)[kKeys]) {
#pragma unroll
  for (int j = 0; j < kKeys; ++j) {
    const int e = lane + 32 * j;
    code[j] = e < E ? static_cast<uint32_t>(topk_key(__ldg(logits + t * E + e), e) >> 32) : 0u;
  }
}

template <int kKeys>
__device__ __forceinline__ void topk_token(uint32_t (&code)[kKeys], int64_t t, int32_t k, int lane,
                                           int32_t* __restrict__ ids, float* __restrict__ w, int32_t* sh_hist) {
  uint32_t best = 0, best_j = 0;
  auto local_best = [&]() {
    best = 0;
    best_j = 0;
#pragma unroll
    for (int j = 0; j < kKeys; ++j)
      if (code[j] > best) {
        best = code[j];
        best_j = j;
      }
  };
  local_best();
  uint32_t mine_code = 0, mine_e = 0;
  for (int s = 0; s < k; ++s) {
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, best);
    const uint32_t e_win = __reduce_min_sync(0xFFFFFFFFu, best == m ? lane + 32u * best_j : 0xFFFFFFFFu);
    if (static_cast<int>(e_win & 31u) == lane) {
#pragma unroll
      for (int j = 0; j < kKeys; ++j)
        if (j == static_cast<int>(e_win >> 5)) code[j] = 0u;
      local_best();
    }
    if (lane == s) {
      mine_code = m;
      mine_e = e_win;
    }
  }
  const uint64_t mine = (static_cast<uint64_t>(mine_code) << 32) | (0xFFFFFFFFu - mine_e);
  // softmax over the selected logits; slot 0 holds the maximum
  const float my_v = key_value(mine);
  const int my_e = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(mine));
  const float mx = __shfl_sync(0xFFFFFFFFu, my_v, 0);
  const float z = lane < k ? expf(my_v - mx) : 0.0f;
  float sum = z;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
  if (lane < k) {
    ids[t * k + lane] = my_e;
    w[t * k + lane] = z / sum;
    atomicAdd(&sh_hist[my_e], 1);
  }
}

template <int kKeys>
__global__ void __launch_bounds__(kTopkThreads) route_topk_kernel(const float* __restrict__ logits, int32_t T,
                                                                  int32_t E, int32_t k, int32_t* __restrict__ ids,
                                                                  float* __restrict__ w,
                                                                  int32_t* __restrict__ chunk_hist) {
  __shared__ int32_t sh_hist[1024];
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh_hist[e] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = kRouteChunk / static_cast<int>(gridDim.y);          // tokens of this block
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kRouteChunk + static_cast<int64_t>(blockIdx.y) * per;
  const int n = static_cast<int>(T - t0 < per ? (T - t0 > 0 ? T - t0 : 0) : per);
  constexpr int kStep = kTopkThreads / 32;
  if (warp < n) {
    uint32_t code[kKeys];
    topk_load<kKeys>(logits, t0 + warp, E, lane, code);
    for (int i = warp; i < n; i += kStep) {
      // the next token's logits are in flight while this one is ranked (up to
      // E = 256; wider rows would not fit twice in registers)
      uint32_t next[kKeys <= 8 ? kKeys : 1];
      if constexpr (kKeys <= 8) {
        if (i + kStep < n) topk_load<kKeys>(logits, t0 + i + kStep, E, lane, next);
      }
      topk_token<kKeys>(code, t0 + i, k, lane, ids, w, sh_hist);
      if constexpr (kKeys <= 8) {
#pragma unroll
        for (int j = 0; j < kKeys; ++j) code[j] = next[j];
      } else {
        if (i + kStep < n) topk_load<kKeys>(logits, t0 + i + kStep, E, lane, code);
      }
    }
  }
  __syncthreads();
  int32_t* row = chunk_hist + static_cast<int64_t>(blockIdx.x) * E;
  if (gridDim.y == 1) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) row[e] = sh_hist[e];
  } else {
    for (int e = threadIdx.x; e < E; e += blockDim.x)
      if (sh_hist[e] != 0) atomicAdd(&row[e], sh_hist[e]);
  }
}

static cudaError_t launch_topk(const RouteBuffers& b, int sms, cudaStream_t stream) {
  const int n_chunks = (b.T + kRouteChunk - 1) / kRouteChunk;
  // a short batch: four blocks per chunk (32 tokens each, one per warp) adding
  // into a cleared histogram, instead of one block walking 128 tokens
  const int split = 4 * n_chunks <= sms ? 4 : 1;
  if (split > 1) {
    const cudaError_t e = cudaMemsetAsync(b.chunk_hist, 0, static_cast<size_t>(n_chunks) * b.E * sizeof(int32_t),
                                          stream);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid(static_cast<unsigned>(n_chunks), static_cast<unsigned>(split)), block(kTopkThreads);
  const int keys = (b.E + 31) / 32;
  if (keys <= 1) route_topk_kernel<1><<<grid, block, 0, stream>>>(b.logits, b.T, b.E, b.top_k, b.topk_ids, b.topk_w, b.chunk_hist);
  else if (keys <= 2) route_topk_kernel<2><<<grid, block, 0, stream>>>(b.logits, b.T, b.E, b.top_k, b.topk_ids, b.topk_w, b.chunk_hist);
  else if (keys <= 4) route_topk_kernel<4><<<grid, block, 0, stream>>>(b.logits, b.T, b.E, b.top_k, b.topk_ids, b.topk_w, b.chunk_hist);
  else if (keys <= 8) route_topk_kernel<8><<<grid, block, 0, stream>>>(b.logits, b.T, b.E, b.top_k, b.topk_ids, b.topk_w, b.chunk_hist);
  else if (keys <= 16) route_topk_kernel<16><<<grid, block, 0, stream>>>(b.logits, b.T, b.E, b.top_k, b.topk_ids, b.topk_w, b.chunk_hist);
  else route_topk_kernel<32><<<grid, block, 0, stream>>>(b.logits, b.T, b.E, b.top_k, b.topk_ids, b.topk_w, b.chunk_hist);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- offsets --
// One block: per expert, turn chunk counts into exclusive per-chunk bases (in
// place) and the total count; then the padded exclusive scan over experts and
// the -1 marks of the padding rows.  The chunk walk is split over P threads per
// expert (P a power of two, P * E <= 1024; thread p + P-ary part q takes a
// contiguous run of chunks), so the walk is P times shorter.
__global__ void __launch_bounds__(1024) route_offsets_kernel(int32_t* __restrict__ chunk_hist,
                                                             int32_t n_chunks, int32_t E,
                                                             int32_t* __restrict__ counts,
                                                             int32_t* __restrict__ offsets,
                                                             int32_t* __restrict__ perm_token) {
  __shared__ int32_t sh_off[1025];
  __shared__ int32_t sh_cnt[1024];
  __shared__ int32_t sh_part[1024];
  __shared__ int32_t sh_warp[32];
  const int tid = threadIdx.x;
  int parts = 1;
  while (parts < 32 && 2 * parts * E <= 1024) parts *= 2;
  const int e = tid % E, q = tid / E;                 // consecutive threads: consecutive experts
  const bool walker = tid < parts * E;
  const int per = (n_chunks + parts - 1) / parts;
  const int c0 = q * per, c1 = c0 + per < n_chunks ? c0 + per : n_chunks;
  int32_t sum = 0;
  if (walker) {
#pragma unroll 8
    for (int c = c0; c < c1; ++c) sum += chunk_hist[static_cast<int64_t>(c) * E + e];
  }
  if (walker) sh_part[tid] = sum;
  __syncthreads();
  if (walker) {
    int32_t run = 0, total = 0;
    for (int r = 0; r < parts; ++r) {
      const int32_t v = sh_part[r * E + e];
      run += r < q ? v : 0;
      total += v;
    }
#pragma unroll 8
    for (int c = c0; c < c1; ++c) {
      const int64_t i = static_cast<int64_t>(c) * E + e;
      const int32_t h = chunk_hist[i];
      chunk_hist[i] = run;
      run += h;
    }
    if (q == 0) {
      counts[e] = total;
      sh_cnt[e] = total;
    }
  }
  __syncthreads();
  const int32_t padded = tid < E ? ((sh_cnt[tid] + 127) / 128) * 128 : 0;
  // block-wide inclusive scan of `padded` (warp shuffles, then warp totals)
  const int lane = tid & 31, warp = tid >> 5;
  int32_t x = padded;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) sh_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int32_t s = sh_warp[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t y = __shfl_up_sync(0xFFFFFFFFu, s, off);
      if (lane >= off) s += y;
    }
    sh_warp[lane] = s;
  }
  __syncthreads();
  const int32_t inclusive = x + (warp > 0 ? sh_warp[warp - 1] : 0);
  if (tid < E) {
    offsets[tid] = inclusive - padded;
    sh_off[tid] = inclusive - padded;
  }
  if (tid == E - 1) {
    offsets[E] = inclusive;
    sh_off[E] = inclusive;
  }
  __syncthreads();
  // padding rows of each group: one warp per expert
  for (int g = warp; g < E; g += 32)
    for (int32_t r = sh_off[g] + sh_cnt[g] + lane; r < sh_off[g + 1]; r += 32) perm_token[r] = -1;
}

// ----------------------------------------------------------------- assign --
// One block per chunk, one thread per token.  A token picks each expert at most
// once, so the rank of (token, expert) among the chunk's rows of that expert is
// the number of earlier tokens of the chunk that picked it: each 32-token group
// sets one bit per token in a per-expert mask, and the rank is the population
// count of the lower bits of its own group's mask plus the full counts of the
// earlier groups' masks.  Rows of an expert therefore come in ascending token order.
constexpr int kAssignGroups = kRouteChunk / 32;

__global__ void __launch_bounds__(kRouteChunk) route_assign_kernel(const int32_t* __restrict__ ids, int32_t T,
                                                                   int32_t E, int32_t k,
                                                                   const int32_t* __restrict__ chunk_base,
                                                                   const int32_t* __restrict__ offsets,
                                                                   int32_t* __restrict__ perm_token,
                                                                   int32_t* __restrict__ inv_perm) {
  extern __shared__ int32_t sh[];
  int32_t* sh_start = sh;                                          // [E] offsets[e] + chunk base
  uint32_t* sh_mask = reinterpret_cast<uint32_t*>(sh + E);         // [kAssignGroups][E]
  const int64_t chunk = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    sh_start[e] = __ldg(offsets + e) + chunk_base[chunk * E + e];
#pragma unroll
    for (int g = 0; g < kAssignGroups; ++g) sh_mask[g * E + e] = 0u;
  }
  __syncthreads();
  const int i = threadIdx.x, g = i >> 5, lane = i & 31;
  const int64_t t = chunk * kRouteChunk + i;
  const bool live = t < T;
  if (live)
    for (int j = 0; j < k; ++j) atomicOr(&sh_mask[g * E + __ldg(ids + t * k + j)], 1u << lane);
  __syncthreads();
  if (live) {
    for (int j = 0; j < k; ++j) {
      const int32_t e = __ldg(ids + t * k + j);
      int32_t rank = __popc(sh_mask[g * E + e] & ((1u << lane) - 1u));
      for (int h = 0; h < g; ++h) rank += __popc(sh_mask[h * E + e]);
      const int32_t row = sh_start[e] + rank;
      perm_token[row] = static_cast<int32_t>(t);
      inv_perm[t * k + j] = row;
    }
  }
}

// ---------------------------------------------------------------- scatter --
constexpr int kPadParts = 4;

// Grid (kPadParts*E + T, ceil(H/1024 / warps)): blocks x < kPadParts*E (with
// y = 0) zero part x % kPadParts of expert x / kPadParts's padding scales, the
// others stage token x - kPadParts*E, one warp per 1024-column segment.
__global__ void __launch_bounds__(256) route_scatter_kernel(const StageJob s) {
  if (blockIdx.x < static_cast<unsigned>(kPadParts * s.E)) {
    if (blockIdx.y == 0) {
      const int part = static_cast<int>(blockIdx.x) % kPadParts;
      stage_padding(s, static_cast<int>(blockIdx.x) / kPadParts, static_cast<int64_t>(part) * blockDim.x + threadIdx.x,
                    static_cast<int64_t>(kPadParts) * blockDim.x);
    }
    return;
  }
  const int64_t segs = (s.H + 1023) / 1024;
  const int64_t seg = static_cast<int64_t>(blockIdx.y) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (seg >= segs) return;
  const int64_t t = static_cast<int64_t>(blockIdx.x) - static_cast<int64_t>(kPadParts) * s.E;
  StageBatch<1> b;
  b.item[0] = t * segs + seg;
  stage_load(s, b, threadIdx.x & 31);
  stage_store(s, b, threadIdx.x & 31);
}

cudaError_t stage_launch(const StageJob& s, cudaStream_t stream) {
  if (s.T == 0) return cudaSuccess;
  const int64_t segs = (s.H + 1023) / 1024;
  const int warps = static_cast<int>(segs < 8 ? segs : 8);     // no idle warps on short rows
  const dim3 grid(static_cast<unsigned>(kPadParts * s.E + s.T), static_cast<unsigned>((segs + warps - 1) / warps));
  route_scatter_kernel<<<grid, 32 * warps, 0, stream>>>(s);
  return cudaGetLastError();
}

cudaError_t route_permute_launch(const RouteBuffers& b, cudaStream_t stream) {
  const int32_t n_chunks = (b.T + kRouteChunk - 1) / kRouteChunk;
  if (n_chunks > 0) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = launch_topk(b, sms, stream);       // every row of the chunk histogram
    if (e != cudaSuccess) return e;
  }
  route_offsets_kernel<<<1, 1024, 0, stream>>>(b.chunk_hist, n_chunks, b.E, b.counts, b.offsets, b.perm_token);
  if (n_chunks > 0) {
    const size_t smem = static_cast<size_t>(b.E) * (1 + kAssignGroups) * sizeof(int32_t);
    route_assign_kernel<<<n_chunks, kRouteChunk, smem, stream>>>(b.topk_ids, b.T, b.E, b.top_k, b.chunk_hist,
                                                                 b.offsets, b.perm_token, b.inv_perm);
    if (b.a1_sf != nullptr) {
      StageJob s;
      s.x = b.x;
      s.x_gscale = b.x_gscale;
      s.inv_perm = b.inv_perm;
      s.counts = b.counts;
      s.offsets = b.offsets;
      s.a_q = b.a1_q;
      s.a_sf = b.a1_sf;
      s.x_q = b.x_q;
      s.T = b.T;
      s.H = b.H;
      s.E = b.E;
      s.k = b.top_k;
      s.rows_max = b.rows_max;
      s.err = device_error_word();
      return stage_launch(s, stream);
    }
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------- combine --
// Block (t, s) of token t takes the 8-column chunks s*blockDim + thread,
// (s + gridDim.y)*blockDim + thread, ...; each thread accumulates its 8 columns
// over the k slots in slot order (fp32 FMA), then the token's shared-expert row
// if there is one, and rounds once to BF16.  Short batches split a token's row
// over several blocks so that enough loads are in flight.  A slot whose row lies
// outside [0, n_rows) loads nothing, adds 0 and sets kErrBounds.
__global__ void __launch_bounds__(128) combine_kernel(const __nv_bfloat16* __restrict__ rows, int64_t n_rows,
                                                      const int32_t* __restrict__ inv_perm,
                                                      const float* __restrict__ w, int32_t H, int32_t k,
                                                      const __nv_bfloat16* __restrict__ shared,
                                                      __nv_bfloat16* __restrict__ y, unsigned* err) {
  const int64_t t = blockIdx.x;
  const int n8 = H / 8;
  for (int c = blockIdx.y * blockDim.x + threadIdx.x; c < n8; c += gridDim.y * blockDim.x) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    // slots in groups of eight: the group's row loads are all issued before the
    // first is used (an index check inside one slot-at-a-time loop kept the
    // compiler from issuing them ahead)
    for (int j0 = 0; j0 < k; j0 += 8) {
      uint4 v[8];
      float wj[8];
      bool in[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        int64_t r = 0;
        wj[q] = 0.0f;
        in[q] = false;
        if (j0 + q < k) {
          r = __ldg(inv_perm + t * k + j0 + q);
          wj[q] = __ldg(w + t * k + j0 + q);
          in[q] = r >= 0 && r < n_rows;
          if (!in[q]) raise_error(err, kErrBounds);
        }
        v[q] = in[q] ? __ldg(reinterpret_cast<const uint4*>(rows + (in[q] ? r : 0) * H) + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (!in[q]) continue;
        float f[8];
        bf16x8_to_f32(v[q], f);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[q], f[i], acc[i]);
      }
    }
    if (shared != nullptr) {
      float v[8];
      bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(shared + t * H) + c), v);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += v[i];
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(y + t * H)[c] = o;
  }
}

cudaError_t combine_launch(const void* rows, int64_t n_rows, const int32_t* inv_perm, const float* w, int32_t T,
                           int32_t H, int32_t top_k, const void* shared, void* y, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  // a token's row over up to ceil(H / 1024) blocks of 128 threads while the batch
  // has fewer than 4096 tokens (one 16-byte chunk per thread)
  const int split = T < 4096 ? (H / 8 + 127) / 128 : 1;
  combine_kernel<<<dim3(T, split), 128, 0, stream>>>(static_cast<const __nv_bfloat16*>(rows), n_rows, inv_perm, w, H,
                                                     top_k, static_cast<const __nv_bfloat16*>(shared),
                                                     static_cast<__nv_bfloat16*>(y), device_error_word());
  return cudaGetLastError();
}

}  // namespace nvfp4

// Routing, padded expert permutation, activation staging and the weighted combine.
//
// "NVFP4 MegaMoE Debug Log", section "NVFP4 MoE Pipeline": stage_activation of
// the hidden states, and the final scatter with routing weights.  "NVFP4-1.1
// Approach, Part 2": the padded per-expert layout (padded_dst gather / scatter).
//
// The permutation is deterministic although it counts with atomics: tokens are
// cut into chunks of kRouteChunk; the top-k kernel counts each chunk's rows per
// expert (atomic increments commute), one block turns the chunk counts into
// per-chunk bases and the 128-padded expert offsets, and each chunk then
// assigns ranks by walking its tokens in order.  Rows of an expert therefore
// come in ascending token order.  x is quantised once per token and the bytes
// are written straight into the token's k permuted rows.
#include <float.h>

#include "common.cuh"
#include "internal.h"

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
// One warp per token: each lane holds the logits of experts lane + 32j and its
// best remaining key; k rounds of a warp max over the lanes' best keys.
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int32_t T,
                                                         int32_t E, int32_t k, int32_t* __restrict__ ids,
                                                         float* __restrict__ w,
                                                         int32_t* __restrict__ chunk_hist) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  uint64_t key[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int e = lane + 32 * j;
    key[j] = e < E ? topk_key(__ldg(logits + t * E + e), e) : 0ull;
  }
  uint32_t taken = 0;
  auto local_best = [&]() {
    uint64_t b = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (!((taken >> j) & 1u) && key[j] > b) b = key[j];
    return b;
  };
  uint64_t best = local_best();
  uint64_t mine = 0;
  for (int s = 0; s < k; ++s) {
    uint64_t m = best;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, m, off);
      m = o > m ? o : m;
    }
    const uint32_t e_win = 0xFFFFFFFFu - static_cast<uint32_t>(m);
    if (static_cast<int>(e_win & 31u) == lane) {
      taken |= 1u << (e_win >> 5);
      best = local_best();
    }
    if (lane == s) mine = m;
  }
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
    atomicAdd(&chunk_hist[(t / kRouteChunk) * E + my_e], 1);
  }
}

// ---------------------------------------------------------------- offsets --
// One block: per expert, turn chunk counts into exclusive per-chunk bases (in
// place) and the total count; then the padded exclusive scan over experts and
// the -1 marks of the padding rows.
__global__ void __launch_bounds__(1024) route_offsets_kernel(int32_t* __restrict__ chunk_hist,
                                                             int32_t n_chunks, int32_t E,
                                                             int32_t* __restrict__ counts,
                                                             int32_t* __restrict__ offsets,
                                                             int32_t* __restrict__ perm_token) {
  __shared__ int32_t sh_off[1025];
  __shared__ int32_t sh_cnt[1024];
  __shared__ int32_t sh_warp[32];
  const int tid = threadIdx.x;
  int32_t padded = 0;
  if (tid < E) {
    int32_t run = 0;
    int32_t c = 0;
    for (; c + 8 <= n_chunks; c += 8) {         // eight independent loads in flight
      int32_t h[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) h[i] = chunk_hist[static_cast<int64_t>(c + i) * E + tid];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        chunk_hist[static_cast<int64_t>(c + i) * E + tid] = run;
        run += h[i];
      }
    }
    for (; c < n_chunks; ++c) {
      const int32_t h = chunk_hist[static_cast<int64_t>(c) * E + tid];
      chunk_hist[static_cast<int64_t>(c) * E + tid] = run;
      run += h;
    }
    counts[tid] = run;
    sh_cnt[tid] = run;
    padded = ((run + 127) / 128) * 128;
  }
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
  for (int e = warp; e < E; e += 32)
    for (int32_t r = sh_off[e] + sh_cnt[e] + lane; r < sh_off[e + 1]; r += 32) perm_token[r] = -1;
}

// ----------------------------------------------------------------- assign --
// One block per chunk: stage the chunk's expert ids, per-chunk bases and the
// offsets in shared memory, then one warp walks the tokens in order; lane j
// places slot j.  A token picks each expert at most once, so the lanes never
// touch the same counter.
__global__ void __launch_bounds__(128) route_assign_kernel(const int32_t* __restrict__ ids, int32_t T,
                                                           int32_t E, int32_t k,
                                                           const int32_t* __restrict__ chunk_base,
                                                           const int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ perm_token,
                                                           int32_t* __restrict__ inv_perm) {
  extern __shared__ int32_t sh[];
  int32_t* sh_local = sh;                // [E] running count per expert
  int32_t* sh_start = sh + E;            // [E] offsets[e] + chunk base
  int32_t* sh_ids = sh + 2 * E;          // [kRouteChunk * k]
  const int64_t chunk = blockIdx.x;
  const int64_t t0 = chunk * kRouteChunk;
  const int n_tok = static_cast<int>(T - t0 < kRouteChunk ? T - t0 : kRouteChunk);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    sh_local[e] = 0;
    sh_start[e] = __ldg(offsets + e) + chunk_base[chunk * E + e];
  }
  for (int i = threadIdx.x; i < n_tok * k; i += blockDim.x) sh_ids[i] = __ldg(ids + t0 * k + i);
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    for (int i = 0; i < n_tok; ++i) {
      if (lane < k) {
        const int32_t e = sh_ids[i * k + lane];
        const int32_t row = sh_start[e] + sh_local[e];
        sh_local[e] += 1;
        perm_token[row] = static_cast<int32_t>(t0 + i);
        inv_perm[(t0 + i) * k + lane] = row;
      }
      __syncwarp();
    }
  }
}

// ---------------------------------------------------------------- scatter --
// Quantise x (PLAIN, per 16 along H) and write the bytes into each of the token's
// k permuted rows.  Grid (T, ceil(H/256 / 8)); one warp per 256-value segment;
// one thread per 8 values, a lane pair per 16-block, a lane octet per scale word.
__global__ void __launch_bounds__(256) route_scatter_kernel(const __nv_bfloat16* __restrict__ x, int32_t H,
                                                            int32_t k, const int32_t* __restrict__ inv_perm,
                                                            uint8_t* __restrict__ a_q,
                                                            uint8_t* __restrict__ a_sf) {
  const int lane = threadIdx.x & 31;
  const int64_t seg = static_cast<int64_t>(blockIdx.y) * 8 + (threadIdx.x >> 5);
  if (seg * 256 >= H) return;
  const int64_t t = blockIdx.x;
  const int64_t c0 = seg * 256 + lane * 8;
  const bool active = c0 < H;
  float h[8];
  if (active) {
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(x + t * H + c0)), h);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] = 0.0f;
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(h[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  const BlockScale s = block_scale(amax);
  const uint32_t nib = quantize8(h, s);
  const uint32_t code = active ? s.code : 0u;
  const int base = lane & ~7;
  const uint32_t word = __shfl_sync(0xFFFFFFFFu, code, base) | (__shfl_sync(0xFFFFFFFFu, code, base + 2) << 8) |
                        (__shfl_sync(0xFFFFFFFFu, code, base + 4) << 16) |
                        (__shfl_sync(0xFFFFFFFFu, code, base + 6) << 24);
  const uint32_t k4 = static_cast<uint32_t>(seg * 4 + (lane >> 3));
  const uint32_t k4_total = static_cast<uint32_t>(H / 64);
  for (int j = 0; j < k; ++j) {
    const int64_t r = __ldg(inv_perm + t * k + j);
    if (active) *reinterpret_cast<uint32_t*>(a_q + r * (H / 2) + c0 / 2) = nib;
    if ((lane & 7) == 0 && k4 < k4_total)
      *reinterpret_cast<uint32_t*>(a_sf + sf_word_offset(r, k4, k4_total)) = word;
  }
}

// -------------------------------------------------------------- pad fill --
// One block per expert: zero the nibbles and scale words of the padding rows
// [offsets[e] + counts[e], offsets[e+1]).
__global__ void __launch_bounds__(256) route_padfill_kernel(const int32_t* __restrict__ counts,
                                                            const int32_t* __restrict__ offsets, int32_t H,
                                                            uint8_t* __restrict__ a_q, uint8_t* __restrict__ a_sf) {
  const int e = blockIdx.x;
  const int64_t lo = __ldg(offsets + e) + __ldg(counts + e);
  const int64_t hi = __ldg(offsets + e + 1);
  const int n16 = H / 32;                 // 16-byte chunks per row
  const int k4_total = H / 64;
  const int64_t nq = (hi - lo) * n16;
  for (int64_t i = threadIdx.x; i < nq; i += blockDim.x) {
    const int64_t r = lo + i / n16;
    reinterpret_cast<uint4*>(a_q + r * (H / 2))[i % n16] = make_uint4(0, 0, 0, 0);
  }
  const int64_t ns = (hi - lo) * k4_total;
  for (int64_t i = threadIdx.x; i < ns; i += blockDim.x) {
    const int64_t r = lo + i / k4_total;
    *reinterpret_cast<uint32_t*>(a_sf + sf_word_offset(r, static_cast<uint32_t>(i % k4_total), k4_total)) = 0u;
  }
}

cudaError_t route_permute_launch(const RouteBuffers& b, cudaStream_t stream) {
  const int32_t n_chunks = (b.T + kRouteChunk - 1) / kRouteChunk;
  if (n_chunks > 0) {
    cudaError_t e = cudaMemsetAsync(b.chunk_hist, 0, static_cast<size_t>(n_chunks) * b.E * sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
    route_topk_kernel<<<(b.T + 7) / 8, 256, 0, stream>>>(b.logits, b.T, b.E, b.top_k, b.topk_ids, b.topk_w,
                                                         b.chunk_hist);
  }
  route_offsets_kernel<<<1, 1024, 0, stream>>>(b.chunk_hist, n_chunks, b.E, b.counts, b.offsets, b.perm_token);
  if (n_chunks > 0) {
    const size_t smem = (2 * static_cast<size_t>(b.E) + static_cast<size_t>(kRouteChunk) * b.top_k) * sizeof(int32_t);
    route_assign_kernel<<<n_chunks, 128, smem, stream>>>(b.topk_ids, b.T, b.E, b.top_k, b.chunk_hist, b.offsets,
                                                         b.perm_token, b.inv_perm);
    route_padfill_kernel<<<b.E, 256, 0, stream>>>(b.counts, b.offsets, b.H, b.a1_q, b.a1_sf);
    const int64_t segs = (b.H + 255) / 256;
    const dim3 grid(static_cast<unsigned>(b.T), static_cast<unsigned>((segs + 7) / 8));
    route_scatter_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(b.x), b.H, b.top_k, b.inv_perm,
                                                   b.a1_q, b.a1_sf);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------- combine --
// One block per token; each thread accumulates 8 columns over the k slots in
// slot order (fp32 FMA) and rounds once to BF16.
__global__ void __launch_bounds__(128) combine_kernel(const __nv_bfloat16* __restrict__ rows,
                                                      const int32_t* __restrict__ inv_perm,
                                                      const float* __restrict__ w, int32_t H, int32_t k,
                                                      __nv_bfloat16* __restrict__ y) {
  const int64_t t = blockIdx.x;
  const int n8 = H / 8;
  for (int c = threadIdx.x; c < n8; c += blockDim.x) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int j = 0; j < k; ++j) {
      const int64_t r = __ldg(inv_perm + t * k + j);
      const float wj = __ldg(w + t * k + j);
      float v[8];
      bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(rows + r * H) + c), v);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, v[i], acc[i]);
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(y + t * H)[c] = o;
  }
}

cudaError_t combine_launch(const void* rows, const int32_t* inv_perm, const float* w, int32_t T, int32_t H,
                           int32_t top_k, void* y, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  combine_kernel<<<T, 128, 0, stream>>>(static_cast<const __nv_bfloat16*>(rows), inv_perm, w, H, top_k,
                                        static_cast<__nv_bfloat16*>(y));
  return cudaGetLastError();
}

}  // namespace nvfp4

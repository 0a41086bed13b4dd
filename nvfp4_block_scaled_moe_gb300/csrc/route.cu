// Routing, padded expert permutation, activation staging and the weighted combine.
//
// "NVFP4 MegaMoE Debug Log", section "NVFP4 MoE Pipeline": stage_activation of
// the hidden states, and the final scatter with routing weights.  "NVFP4-1.1
// Approach, Part 2": the padded per-expert layout (padded_dst gather / scatter).
//
// The permutation is deterministic without ordered atomics: tokens are cut into
// chunks of kRouteChunk; each chunk counts its rows per expert (order-free
// shared-memory atomics), one block turns the chunk counts into per-chunk bases
// and the 128-padded expert offsets, and each chunk then assigns ranks by
// walking its tokens in order.  Rows of an expert therefore come in ascending
// token order.
#include <float.h>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

// ------------------------------------------------------------------ top-k --
// One block per chunk of kRouteChunk tokens, 8 warps, one warp per token at a time.
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int32_t T,
                                                         int32_t E, int32_t k, int32_t* __restrict__ ids,
                                                         float* __restrict__ w,
                                                         int32_t* __restrict__ chunk_hist) {
  extern __shared__ int32_t sh_count[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh_count[e] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t chunk = blockIdx.x;
  for (int i = warp; i < kRouteChunk; i += 8) {
    const int64_t t = chunk * kRouteChunk + i;
    if (t >= T) break;
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int e = lane + 32 * j;
      v[j] = e < E ? __ldg(logits + t * E + e) : -FLT_MAX;
    }
    uint32_t taken = 0;
    float my_v = 0.0f;
    int my_e = 0;
    for (int s = 0; s < k; ++s) {
      float best_v = -INFINITY;
      int best_e = INT32_MAX;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int e = lane + 32 * j;
        if (e < E && !((taken >> j) & 1u) && (v[j] > best_v || (v[j] == best_v && e < best_e))) {
          best_v = v[j];
          best_e = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, best_v, off);
        const int oe = __shfl_xor_sync(0xFFFFFFFFu, best_e, off);
        if (ov > best_v || (ov == best_v && oe < best_e)) {
          best_v = ov;
          best_e = oe;
        }
      }
      if ((best_e & 31) == lane) taken |= 1u << (best_e >> 5);
      if (lane == s) {
        my_v = best_v;
        my_e = best_e;
      }
    }
    // softmax over the selected logits; slot 0 holds the maximum
    const float mx = __shfl_sync(0xFFFFFFFFu, my_v, 0);
    const float z = lane < k ? expf(my_v - mx) : 0.0f;
    float sum = z;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
    if (lane < k) {
      ids[t * k + lane] = my_e;
      w[t * k + lane] = z / sum;
      atomicAdd(&sh_count[my_e], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_hist[chunk * E + e] = sh_count[e];
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
  __shared__ int32_t sh_pad[1024];
  __shared__ int32_t sh_warp[32];
  const int tid = threadIdx.x;
  int32_t padded = 0;
  if (tid < E) {
    int32_t run = 0;
    for (int32_t c = 0; c < n_chunks; ++c) {
      const int32_t h = chunk_hist[static_cast<int64_t>(c) * E + tid];
      chunk_hist[static_cast<int64_t>(c) * E + tid] = run;
      run += h;
    }
    counts[tid] = run;
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
  const int32_t exclusive = inclusive - padded;
  if (tid < E) {
    offsets[tid] = exclusive;
    sh_pad[tid] = exclusive;
  }
  if (tid == E - 1) offsets[E] = inclusive;
  __syncthreads();
  // padding rows of each group
  for (int e = 0; e < E; ++e) {
    const int32_t lo = sh_pad[e] + counts[e];
    const int32_t hi = (e + 1 < E) ? sh_pad[e + 1] : offsets[E];
    for (int32_t r = lo + tid; r < hi; r += blockDim.x) perm_token[r] = -1;
  }
}

// ----------------------------------------------------------------- assign --
// One warp per chunk: walk the chunk's tokens in order; lane j places slot j.
// A token picks each expert at most once, so the lanes never touch the same counter.
__global__ void __launch_bounds__(32) route_assign_kernel(const int32_t* __restrict__ ids, int32_t T,
                                                          int32_t E, int32_t k,
                                                          const int32_t* __restrict__ chunk_base,
                                                          const int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ perm_token,
                                                          int32_t* __restrict__ inv_perm) {
  extern __shared__ int32_t sh_local[];
  const int lane = threadIdx.x;
  const int64_t chunk = blockIdx.x;
  for (int e = lane; e < E; e += 32) sh_local[e] = 0;
  __syncwarp();
  for (int i = 0; i < kRouteChunk; ++i) {
    const int64_t t = chunk * kRouteChunk + i;
    if (t >= T) break;
    if (lane < k) {
      const int32_t e = ids[t * k + lane];
      const int32_t rank = chunk_base[chunk * E + e] + sh_local[e];
      sh_local[e] += 1;
      const int32_t row = offsets[e] + rank;
      perm_token[row] = static_cast<int32_t>(t);
      inv_perm[t * k + lane] = row;
    }
    __syncwarp();
  }
}

// ----------------------------------------------------------------- gather --
// One warp per padded row below offsets[E]: copy the staged NVFP4 row of its
// token (16-byte chunks) and its scale words into the swizzled layout; padding
// rows get zeros.
__global__ void __launch_bounds__(256) route_gather_kernel(const int32_t* __restrict__ perm_token,
                                                           const int32_t* __restrict__ offsets, int32_t E,
                                                           int64_t rows_max, int32_t H,
                                                           const uint8_t* __restrict__ x_q,
                                                           const uint8_t* __restrict__ x_sf,
                                                           uint8_t* __restrict__ a_q, uint8_t* __restrict__ a_sf) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (row >= rows_max || row >= __ldg(offsets + E)) return;
  const int32_t t = __ldg(perm_token + row);
  const int n16 = H / 32;          // 16-byte chunks per row of H/2 bytes
  uint4* dst = reinterpret_cast<uint4*>(a_q + row * (H / 2));
  if (t >= 0) {
    const uint4* src = reinterpret_cast<const uint4*>(x_q + static_cast<int64_t>(t) * (H / 2));
    for (int c = lane; c < n16; c += 32) dst[c] = __ldg(src + c);
  } else {
    for (int c = lane; c < n16; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
  }
  const int k4_total = H / 64;
  const uint32_t* sw = reinterpret_cast<const uint32_t*>(x_sf + static_cast<int64_t>(t < 0 ? 0 : t) * (H / 16));
  for (int w = lane; w < k4_total; w += 32) {
    const uint32_t word = t >= 0 ? __ldg(sw + w) : 0u;
    *reinterpret_cast<uint32_t*>(a_sf + sf_word_offset(row, w, k4_total)) = word;
  }
}

cudaError_t route_permute_launch(const RouteBuffers& b, cudaStream_t stream) {
  const int32_t n_chunks = (b.T + kRouteChunk - 1) / kRouteChunk;
  const size_t hist_smem = static_cast<size_t>(b.E) * sizeof(int32_t);
  if (n_chunks > 0) {
    route_topk_kernel<<<n_chunks, 256, hist_smem, stream>>>(b.logits, b.T, b.E, b.top_k, b.topk_ids, b.topk_w,
                                                            b.chunk_hist);
  }
  route_offsets_kernel<<<1, 1024, 0, stream>>>(b.chunk_hist, n_chunks, b.E, b.counts, b.offsets, b.perm_token);
  if (n_chunks > 0) {
    route_assign_kernel<<<n_chunks, 32, hist_smem, stream>>>(b.topk_ids, b.T, b.E, b.top_k, b.chunk_hist,
                                                             b.offsets, b.perm_token, b.inv_perm);
    cudaError_t e = quantize_launch(b.x, NVFP4_IN_BF16, NVFP4_MODE_PLAIN, b.T, b.H, b.H, b.x_q, b.x_sf,
                                    /*sf_linear=*/1, nullptr, stream);
    if (e != cudaSuccess) return e;
    const int64_t warps = b.rows_max;
    route_gather_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, stream>>>(
        b.perm_token, b.offsets, b.E, b.rows_max, b.H, b.x_q, b.x_sf, b.a1_q, b.a1_sf);
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

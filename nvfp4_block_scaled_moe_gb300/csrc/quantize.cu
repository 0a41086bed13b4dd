// Standalone NVFP4 quantiser (plain and SwiGLU-of-interleaved-gate/up modes)
// and the scale-factor swizzle.
//
// "NVFP4-1.1 Approach, Part 2": the quantize_nvfp4 kernel (BF16 -> packed E2M1 +
// E4M3 per 16) and the deinterleave + quantise kernel that reads L1 output
// interleaved at granularity 8.  Here the SwiGLU mode computes silu(g) * u from
// each gate/up pair in the same pass.  "NVFP4 MegaMoE Debug Log": the SF remap
// (forward mapping with explicit source strides) for the swizzle kernel.
//
// Layout of the quantiser's work: one thread owns one 16-block (32 bytes of BF16,
// 64 of fp32 or gate+up), a lane quad owns one 64-column group, whose four scale
// bytes form one 32-bit word of the swizzled layout.
//
// Two-level scale ("NVFP4 MoE Pipeline": stage_activation returns an
// input_global_scale next to the per-16 scales): with an encode scale g the
// quantised values are fp32(v * g); nvfp4_global_scale computes g = 2688 / amax
// (6 x 448, the top of the E2M1 x E4M3 range) in two launches.
#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

// Load the 16 values of output block c0 .. c0+15 (c0 % 16 == 0) of a row.
template <int kMode, int kDtype>
__device__ __forceinline__ void load_block(const void* in, int64_t row, int64_t ld, int64_t c0, float (&h)[16]) {
  if (kMode == NVFP4_MODE_SWIGLU_GU8) {
    // interleaved columns 2*c0 .. 2*c0+31: g0(8) u0(8) g1(8) u1(8)
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(in) + row * ld + 2 * c0);
    const uint4 g0 = __ldg(p), u0 = __ldg(p + 1), g1 = __ldg(p + 2), u1 = __ldg(p + 3);
    float g[8], u[8];
    bf16x8_to_f32(g0, g);
    bf16x8_to_f32(u0, u);
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      const float2 t = swiglu2(make_float2(g[i], g[i + 1]), make_float2(u[i], u[i + 1]));
      h[i] = t.x;
      h[i + 1] = t.y;
    }
    bf16x8_to_f32(g1, g);
    bf16x8_to_f32(u1, u);
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      const float2 t = swiglu2(make_float2(g[i], g[i + 1]), make_float2(u[i], u[i + 1]));
      h[8 + i] = t.x;
      h[8 + i + 1] = t.y;
    }
  } else if (kMode == NVFP4_MODE_DEINTERLEAVE_GU8) {
    // interleaved columns 2*c0 .. 2*c0+31: keep u0(8) and u1(8) as they are
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(in) + row * ld + 2 * c0);
    float lo[8], hi[8];
    bf16x8_to_f32(__ldg(p + 1), lo);
    bf16x8_to_f32(__ldg(p + 3), hi);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      h[i] = lo[i];
      h[8 + i] = hi[i];
    }
  } else if (kDtype == NVFP4_IN_BF16) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(in) + row * ld + c0);
    float lo[8], hi[8];
    bf16x8_to_f32(__ldg(p), lo);
    bf16x8_to_f32(__ldg(p + 1), hi);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      h[i] = lo[i];
      h[8 + i] = hi[i];
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(in) + row * ld + c0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v = __ldg(p + q);
      h[4 * q] = v.x;
      h[4 * q + 1] = v.y;
      h[4 * q + 2] = v.z;
      h[4 * q + 3] = v.w;
    }
  }
}

// One thread per 16-block (no shuffle for the amax; one block scale per thread),
// one warp per 512-column segment: blockIdx.x is the row (rows_pad >= rows
// covers the zero padding rows of the swizzled SF), blockIdx.y * (warps per
// block) + warp the segment.  Lanes 4w .. 4w+3 own one 64-column group, whose four scale bytes form
// one 32-bit word of the swizzled layout.  sf_linear selects a plain row-major
// SF output ([rows, cols/16]; requires cols % 64 == 0).
template <int kMode, int kDtype, bool kScaled>
__global__ void __launch_bounds__(256) quantize_kernel(const void* __restrict__ in, int64_t rows,
                                                       int64_t cols, int64_t ld, int64_t rows_pad,
                                                       uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                       int sf_linear, const float* __restrict__ gscale,
                                                       float* __restrict__ h_dbg) {
  const int lane = threadIdx.x & 31;
  const int64_t seg = static_cast<int64_t>(blockIdx.y) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (seg * 512 >= cols) return;
  const int64_t row = blockIdx.x;
  const int64_t c0 = seg * 512 + lane * 16;
  const bool in_row = row < rows;
  const bool active = in_row && c0 < cols;

  float h[16];
  if (active) {
    load_block<kMode, kDtype>(in, row, ld, c0, h);
    if (h_dbg != nullptr) {
      float4* hp = reinterpret_cast<float4*>(h_dbg + row * cols + c0);
#pragma unroll
      for (int i = 0; i < 4; ++i) hp[i] = make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
    }
    if (kScaled) {
      const float g = __ldg(gscale);
#pragma unroll
      for (int i = 0; i < 16; ++i) h[i] *= g;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) h[i] = 0.0f;
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(h[i]));
  const BlockScale s = block_scale(amax);

  if (active) {
    float lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      lo[i] = h[i];
      hi[i] = h[8 + i];
    }
    *reinterpret_cast<uint2*>(q + row * (cols / 2) + c0 / 2) = make_uint2(quantize8(lo, s), quantize8(hi, s));
  }

  // gather the quad's four scale bytes (lanes 4w .. 4w+3) into one word at lane 4w
  const uint32_t code = active ? s.code : 0u;
  const uint32_t word = code | (__shfl_down_sync(0xFFFFFFFFu, code, 1) << 8) |
                        (__shfl_down_sync(0xFFFFFFFFu, code, 2) << 16) |
                        (__shfl_down_sync(0xFFFFFFFFu, code, 3) << 24);
  const int64_t k4 = seg * 8 + (lane >> 2);          // 64-column group of this quad
  const int64_t k4_total = (cols + 63) / 64;
  if ((lane & 3) == 0 && k4 < k4_total) {
    if (sf_linear) {
      if (in_row) *reinterpret_cast<uint32_t*>(sf + row * (cols / 16) + k4 * 4) = word;
    } else {
      *reinterpret_cast<uint32_t*>(sf + sf_word_offset(row, k4, k4_total)) = word;
    }
  }
}

template <int kMode, int kDtype>
static cudaError_t launch_quantize(const void* in, int64_t rows, int64_t cols, int64_t ld,
                                   int64_t rows_pad, uint8_t* q, uint8_t* sf, int sf_linear,
                                   const float* gscale, float* h_dbg, cudaStream_t stream) {
  const int64_t segs = (cols + 511) / 512;
  if (rows_pad == 0) return cudaSuccess;
  const int warps = static_cast<int>(segs < 8 ? segs : 8);      // no idle warps on short rows
  const dim3 grid(static_cast<unsigned>(rows_pad), static_cast<unsigned>((segs + warps - 1) / warps));
  if (gscale != nullptr)
    quantize_kernel<kMode, kDtype, true><<<grid, 32 * warps, 0, stream>>>(in, rows, cols, ld, rows_pad, q, sf,
                                                                          sf_linear, gscale, h_dbg);
  else
    quantize_kernel<kMode, kDtype, false><<<grid, 32 * warps, 0, stream>>>(in, rows, cols, ld, rows_pad, q, sf,
                                                                           sf_linear, nullptr, h_dbg);
  return cudaGetLastError();
}

cudaError_t quantize_launch(const void* in, int dtype, int mode, int64_t rows, int64_t cols, int64_t ld,
                            uint8_t* q, uint8_t* sf, int sf_linear, const float* gscale, float* h_dbg,
                            cudaStream_t stream) {
  const int64_t rows_pad = sf_linear ? rows : ((rows + 127) / 128) * 128;
  if (mode == NVFP4_MODE_SWIGLU_GU8)
    return launch_quantize<NVFP4_MODE_SWIGLU_GU8, NVFP4_IN_BF16>(in, rows, cols, ld, rows_pad, q, sf,
                                                                 sf_linear, gscale, h_dbg, stream);
  if (mode == NVFP4_MODE_DEINTERLEAVE_GU8)
    return launch_quantize<NVFP4_MODE_DEINTERLEAVE_GU8, NVFP4_IN_BF16>(in, rows, cols, ld, rows_pad, q, sf,
                                                                       sf_linear, gscale, h_dbg, stream);
  if (dtype == NVFP4_IN_BF16)
    return launch_quantize<NVFP4_MODE_PLAIN, NVFP4_IN_BF16>(in, rows, cols, ld, rows_pad, q, sf, sf_linear,
                                                            gscale, h_dbg, stream);
  return launch_quantize<NVFP4_MODE_PLAIN, NVFP4_IN_F32>(in, rows, cols, ld, rows_pad, q, sf, sf_linear,
                                                         gscale, h_dbg, stream);
}

// ---------------------------------------------------------- global scale --
// amax over a rows x cols matrix (row stride ld): grid-stride over 8-value
// chunks, four independent 16-byte loads in flight per thread per step, a block
// max, one atomicMax on the float bits (non-negative floats order like their
// bit patterns) into *out, which the launcher zeroed.
template <int kDtype, bool kContig>
__device__ __forceinline__ float chunk_amax(const void* in, int64_t i, int64_t chunks_per_row, int64_t ld) {
  // contiguous rows (ld == cols): chunk i starts at element 8i, no division
  const int64_t r = kContig ? 0 : i / chunks_per_row;
  const int64_t c = kContig ? 8 * i : (i - r * chunks_per_row) * 8;
  float v[8];
  if (kDtype == NVFP4_IN_BF16) {
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(in) + r * ld + c)), v);
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(in) + r * ld + c);
    const float4 a = __ldg(p), b = __ldg(p + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  float m = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[j]));
  return m;
}

template <int kDtype, bool kContig>
__global__ void __launch_bounds__(256) tensor_amax_kernel(const void* __restrict__ in, int64_t rows, int64_t cols,
                                                          int64_t ld, unsigned* __restrict__ out) {
  const int64_t chunks_per_row = cols / 8;
  const int64_t n = rows * chunks_per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  float m = 0.0f;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const float m0 = chunk_amax<kDtype, kContig>(in, i, chunks_per_row, ld);
    const float m1 = chunk_amax<kDtype, kContig>(in, i + stride, chunks_per_row, ld);
    const float m2 = chunk_amax<kDtype, kContig>(in, i + 2 * stride, chunks_per_row, ld);
    const float m3 = chunk_amax<kDtype, kContig>(in, i + 3 * stride, chunks_per_row, ld);
    m = fmaxf(m, fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)));
  }
  for (; i < n; i += stride) m = fmaxf(m, chunk_amax<kDtype, kContig>(in, i, chunks_per_row, ld));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  __shared__ float warp_max[8];
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.0f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) b = fmaxf(b, warp_max[w]);
    atomicMax(out, __float_as_uint(b));
  }
}

// *g = 2688 / amax (IEEE quotient), or 1 when amax is 0 or the quotient is not finite.
__global__ void global_scale_finalize_kernel(float* g) {
  const float amax = __uint_as_float(*reinterpret_cast<const unsigned*>(g));
  float v = amax > 0.0f ? __fdiv_rn(2688.0f, amax) : 1.0f;
  if (!isfinite(v)) v = 1.0f;
  *g = v;
}

cudaError_t global_scale_launch(const void* in, int dtype, int64_t rows, int64_t cols, int64_t ld, float* g_out,
                                int sms, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(g_out, 0, sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const int64_t n = rows * (cols / 8);
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 152) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  unsigned* acc = reinterpret_cast<unsigned*>(g_out);
  const dim3 grid(static_cast<unsigned>(blocks));
  if (ld == cols) {
    if (dtype == NVFP4_IN_BF16)
      tensor_amax_kernel<NVFP4_IN_BF16, true><<<grid, 256, 0, stream>>>(in, rows, cols, ld, acc);
    else
      tensor_amax_kernel<NVFP4_IN_F32, true><<<grid, 256, 0, stream>>>(in, rows, cols, ld, acc);
  } else {
    if (dtype == NVFP4_IN_BF16)
      tensor_amax_kernel<NVFP4_IN_BF16, false><<<grid, 256, 0, stream>>>(in, rows, cols, ld, acc);
    else
      tensor_amax_kernel<NVFP4_IN_F32, false><<<grid, 256, 0, stream>>>(in, rows, cols, ld, acc);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  global_scale_finalize_kernel<<<1, 1, 0, stream>>>(g_out);
  return cudaGetLastError();
}

// ------------------------------------------------------------ SF swizzle --
// Forward: one thread per 32-bit word of the swizzled buffer (row, k4), reading
// four strided source bytes (zero outside mn_rows x k_sf_cols).
__global__ void sf_swizzle_fwd_kernel(const uint8_t* __restrict__ lin, int64_t mn_rows, int64_t k_sf,
                                      int64_t s_mn, int64_t s_k, uint8_t* __restrict__ swz,
                                      int64_t rows_pad, int64_t k4_total) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= rows_pad * k4_total) return;
  const int64_t row = i / k4_total;
  const int64_t k4 = i - row * k4_total;
  uint32_t word = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int64_t k = k4 * 4 + j;
    if (row < mn_rows && k < k_sf) word |= static_cast<uint32_t>(lin[row * s_mn + k * s_k]) << (8 * j);
  }
  *reinterpret_cast<uint32_t*>(swz + sf_word_offset(row, static_cast<uint32_t>(k4), static_cast<uint32_t>(k4_total))) = word;
}

// Inverse: one thread per addressed scale.
__global__ void sf_swizzle_inv_kernel(const uint8_t* __restrict__ swz, int64_t mn_rows, int64_t k_sf,
                                      int64_t s_mn, int64_t s_k, uint8_t* __restrict__ lin,
                                      int64_t k4_total) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= mn_rows * k_sf) return;
  const int64_t row = i / k_sf;
  const int64_t k = i - row * k_sf;
  const uint64_t off = sf_word_offset(row, static_cast<uint32_t>(k >> 2), static_cast<uint32_t>(k4_total)) + (k & 3);
  lin[row * s_mn + k * s_k] = swz[off];
}

cudaError_t sf_swizzle_launch(const uint8_t* in, int64_t mn_rows, int64_t k_sf, int64_t s_mn, int64_t s_k,
                              uint8_t* out, int inverse, cudaStream_t stream) {
  const int64_t k4_total = (k_sf + 3) / 4;
  if (!inverse) {
    const int64_t rows_pad = ((mn_rows + 127) / 128) * 128;
    const int64_t n = rows_pad * k4_total;
    sf_swizzle_fwd_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
        in, mn_rows, k_sf, s_mn, s_k, out, rows_pad, k4_total);
  } else {
    const int64_t n = mn_rows * k_sf;
    sf_swizzle_inv_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
        in, mn_rows, k_sf, s_mn, s_k, out, k4_total);
  }
  return cudaGetLastError();
}

}  // namespace nvfp4

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
    for (int i = 0; i < 8; ++i) h[i] = swiglu(g[i], u[i]);
    bf16x8_to_f32(g1, g);
    bf16x8_to_f32(u1, u);
#pragma unroll
    for (int i = 0; i < 8; ++i) h[8 + i] = swiglu(g[i], u[i]);
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
template <int kMode, int kDtype>
__global__ void __launch_bounds__(256) quantize_kernel(const void* __restrict__ in, int64_t rows,
                                                       int64_t cols, int64_t ld, int64_t rows_pad,
                                                       uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                       int sf_linear, float* __restrict__ h_dbg) {
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
    if (h_dbg != nullptr) {
      float4* hp = reinterpret_cast<float4*>(h_dbg + row * cols + c0);
#pragma unroll
      for (int i = 0; i < 4; ++i) hp[i] = make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
    }
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
                                   float* h_dbg, cudaStream_t stream) {
  const int64_t segs = (cols + 511) / 512;
  if (rows_pad == 0) return cudaSuccess;
  const int warps = static_cast<int>(segs < 8 ? segs : 8);      // no idle warps on short rows
  const dim3 grid(static_cast<unsigned>(rows_pad), static_cast<unsigned>((segs + warps - 1) / warps));
  quantize_kernel<kMode, kDtype><<<grid, 32 * warps, 0, stream>>>(in, rows, cols, ld, rows_pad, q, sf, sf_linear,
                                                                  h_dbg);
  return cudaGetLastError();
}

cudaError_t quantize_launch(const void* in, int dtype, int mode, int64_t rows, int64_t cols, int64_t ld,
                            uint8_t* q, uint8_t* sf, int sf_linear, float* h_dbg, cudaStream_t stream) {
  const int64_t rows_pad = sf_linear ? rows : ((rows + 127) / 128) * 128;
  if (mode == NVFP4_MODE_SWIGLU_GU8)
    return launch_quantize<NVFP4_MODE_SWIGLU_GU8, NVFP4_IN_BF16>(in, rows, cols, ld, rows_pad, q, sf,
                                                                 sf_linear, h_dbg, stream);
  if (dtype == NVFP4_IN_BF16)
    return launch_quantize<NVFP4_MODE_PLAIN, NVFP4_IN_BF16>(in, rows, cols, ld, rows_pad, q, sf, sf_linear,
                                                            h_dbg, stream);
  return launch_quantize<NVFP4_MODE_PLAIN, NVFP4_IN_F32>(in, rows, cols, ld, rows_pad, q, sf, sf_linear,
                                                         h_dbg, stream);
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

// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "nvfp4moe.h"

namespace nvfp4 {

// per-device error word (abi.cu): device address for the current device
unsigned* device_error_word();

cudaError_t quantize_launch(const void* in, int dtype, int mode, int64_t rows, int64_t cols, int64_t ld,
                            uint8_t* q, uint8_t* sf, int sf_linear, const float* gscale, float* h_dbg,
                            cudaStream_t stream);

// g_out = 2688 / amax over the matrix (1 for an all-zero one); cols % 8 == 0.
cudaError_t global_scale_launch(const void* in, int dtype, int64_t rows, int64_t cols, int64_t ld, float* g_out,
                                int sms, cudaStream_t stream);

cudaError_t sf_swizzle_launch(const uint8_t* in, int64_t mn_rows, int64_t k_sf, int64_t s_mn, int64_t s_k,
                              uint8_t* out, int inverse, cudaStream_t stream);

struct RouteBuffers {
  const float* logits;
  const void* x;
  int32_t T, H, E, top_k;
  int32_t* topk_ids;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm_token;
  int32_t* inv_perm;
  uint8_t* a1_q;           // permuted rows (null: not written)
  uint8_t* a1_sf;
  uint8_t* x_q;            // token-order rows of x (null: not written)
  const float* x_gscale;   // two-level encode scale of x (device scalar) or null
  int64_t rows_max;
  int32_t* chunk_hist;   // workspace: [n_chunks, E] expert counts per token chunk
};

constexpr int kRouteChunk = 128;   // tokens per routing chunk

// Workspace bytes of moe_route_permute and its carve-up (the chunk histogram).
size_t route_workspace_bytes(int32_t T, int32_t E);
void route_carve_workspace(RouteBuffers& b, void* workspace);

// Routing, and the activation staging when b.a1_sf is set.
cudaError_t route_permute_launch(const RouteBuffers& b, cudaStream_t stream);

// The activation staging of a routed batch: x quantised once per token (per 16
// along H, optionally after the two-level scale) and its bytes written into
// each of the token's k permuted rows of a_q / a_sf; the padding rows of every
// expert get zero scale words.  T == 0: nothing.
struct StageJob {
  const void* x;              // [T, H] BF16
  const float* x_gscale;      // two-level encode scale of x (device scalar) or null
  const int32_t* inv_perm;    // [T, k]
  const int32_t* counts;      // [E]
  const int32_t* offsets;     // [E + 1]
  uint8_t* a_q;               // permuted rows (null: not written)
  uint8_t* a_sf;              // their swizzled scales
  uint8_t* x_q;               // token-order rows of x (null: not written)
  int32_t T, H, E, k;
  int64_t rows_max;           // rows of a_q / a_sf: rows outside are not written (error word)
  unsigned* err;              // the device error word
};

cudaError_t stage_launch(const StageJob& s, cudaStream_t stream);

// n_rows: rows of `rows`; a slot outside [0, n_rows) adds 0 and sets the error word
cudaError_t combine_launch(const void* rows, int64_t n_rows, const int32_t* inv_perm, const float* w, int32_t T,
                           int32_t H, int32_t top_k, const void* shared, void* y, cudaStream_t stream);

struct GemmArgs {
  const uint8_t* a_q;
  const uint8_t* a_sf;
  int64_t rows_max;
  const int32_t* a_gather;  // null, or the a_q row of every padded row (< 0: a zero-scale row)
  int64_t a_rows;           // rows of a_q under a gather index
  const int32_t* offsets;
  const int32_t* counts;
  int32_t G, N, K;
  const uint8_t* b_q;
  const uint8_t* b_sf;
  float alpha;
  const float* a_gscale;   // two-level encode scales (device): A's scalar, B's per group,
  const float* b_gscale;   // and the SwiGLU output's scalar; null = 1
  const float* out_gscale;
  int epilogue;
  uint8_t* out_q;
  uint8_t* out_sf;
  void* out_bf16;
  float* h_debug;
  // side job of the CTA-pair SwiGLU kernel: the combine of an earlier batch
  // (moe_combine without shared rows); side_T == 0: none
  const void* side_rows = nullptr;
  int64_t side_n_rows = 0;    // rows of side_rows (index check)
  const int32_t* side_inv = nullptr;
  const float* side_w = nullptr;
  void* side_y = nullptr;
  int32_t side_T = 0, side_H = 0, side_k = 0;
  // side job of the CTA-pair BF16 kernel: the activation staging of a later
  // batch (x_q null); stage.T == 0: none
  StageJob stage = {};
};

// Returns a status; writes a message with set_error_message on failure.
nvfp4_status gemm_launch(const GemmArgs& a, cudaStream_t stream);
// The CTA-pair kernel (N % 256 == 0, at most kPairMaxGroups groups); sms and
// dev of the current device.  left_ctas > 0: a split (common.cuh:
// leftover_split) whose single-CTA launch of left_ctas CTAs the caller makes
// beside this one; the launch leaves their SMs free and returns its cluster
// count in *clusters_out.
constexpr int kPairMaxGroups = 512;
nvfp4_status gemm_pair_launch(const GemmArgs& a, int sms, int dev, cudaStream_t stream, int left_ctas = 0,
                              int* clusters_out = nullptr);
nvfp4_status set_gemm_tiles(int mode);

// 2-D tensor map of a row-major rows x cols matrix (gemm.cu).
bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t rows, uint64_t cols,
                  uint32_t elem_bytes, uint32_t box_cols, uint32_t box_rows, bool swizzle128);

cudaError_t selftest_wait_launch(const int32_t* flag, int64_t limit_ns, cudaStream_t stream);

// error-message helpers (abi.cu)
nvfp4_status fail(nvfp4_status st, const char* fmt, ...);
nvfp4_status fail_cuda(cudaError_t e, const char* where);

}  // namespace nvfp4

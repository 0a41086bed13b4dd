// moe_route_permute_static: moe_route_permute without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they route
// tokens: an inference engine that hands out all memory from its own pool up
// front, code running under a custom allocator that must not see extra
// allocations, or a host path that is not allowed to call cudaMalloc (which can
// synchronise the device) in the middle of a step.  For them this entry point
// keeps the routing scratch (the per-chunk expert histograms) in one
// file-scope device array of kStaticScratchBytes, which the
// CUDA module reserves on every GPU that loads the library for the life of the
// process.  The entry point itself calls no cudaMalloc, cudaFree or allocating
// library routine.
//
// Rules for callers:
//   * the scratch limit: moe_route_permute_workspace(T, H, E, top_k) must not
//     exceed kStaticScratchBytes (16 MiB: ceil(T/128) * E * 4 bytes, e.g. up to
//     about 2 million tokens at E = 256); larger problems are rejected with
//     NVFP4_ERR_UNSUPPORTED;
//   * every call on a device shares the one array and leaves its contents
//     behind; each call clears the histogram it uses before counting, so no
//     state leaks between calls, but calls that overlap on the GPU (on two
//     streams, or from two host threads without ordering) race on the array;
//   * the first call on each device looks up the array's device address with
//     cudaGetSymbolAddress (with that device current); make that first call
//     before any stream capture.  The address is kept for the life of the
//     process: after cudaDeviceReset on a device the library's module is loaded
//     anew, so this entry point must not be used on that device again (the
//     per-device error word of the other calls is cached the same way).
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;

static __device__ __align__(256) uint8_t g_route_scratch[kStaticScratchBytes];

// Device address of g_route_scratch on the current device (looked up once per device).
static nvfp4_status static_scratch(uint8_t** out) {
  static uint8_t* addr[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "moe_route_permute_static: cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(NVFP4_ERR_UNSUPPORTED, "moe_route_permute_static: device %d", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return fail_cuda(e, "moe_route_permute_static: cudaGetSymbolAddress");
    addr[dev] = static_cast<uint8_t*>(p);
  }
  *out = addr[dev];
  return NVFP4_OK;
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status moe_route_permute_static(const float* logits, const void* x_bf16, int32_t T, int32_t H,
                                                  int32_t E, int32_t top_k, int32_t* topk_ids, float* topk_w,
                                                  int32_t* expert_counts, int32_t* expert_offsets,
                                                  int32_t* perm_token, int32_t* inv_perm, uint8_t* a1_q,
                                                  uint8_t* a1_sf, uint8_t* x_q, const float* x_global_scale,
                                                  nvfp4_stream_t stream) {
  if (T < 0) return fail(NVFP4_ERR_INVALID_ARG, "moe_route_permute_static: T=%d", T);
  if (!expert_counts || !expert_offsets)
    return fail(NVFP4_ERR_INVALID_ARG, "moe_route_permute_static: null pointer");
  if (T > 0 && !(logits && topk_ids && topk_w && perm_token && inv_perm))
    return fail(NVFP4_ERR_INVALID_ARG, "moe_route_permute_static: null pointer");
  // a1_sf NULL: routing only (a1_q and x_q NULL too); else x and a1_q and / or x_q
  if (T > 0 && !(a1_sf ? (x_bf16 && (a1_q || x_q)) : (!a1_q && !x_q)))
    return fail(NVFP4_ERR_INVALID_ARG,
                "moe_route_permute_static: staging needs x, a1_sf and a1_q or x_q (routing only: all four NULL)");
  if (E < 1 || E > 1024) return fail(NVFP4_ERR_UNSUPPORTED, "moe_route_permute_static: E=%d outside [1, 1024]", E);
  if (top_k < 1 || top_k > E || top_k > 32)
    return fail(NVFP4_ERR_UNSUPPORTED, "moe_route_permute_static: top_k=%d outside [1, min(E, 32)]", top_k);
  if (H <= 0 || H % 64 != 0)
    return fail(NVFP4_ERR_UNSUPPORTED, "moe_route_permute_static: H=%d is not a positive multiple of 64", H);
  const uintptr_t mis = reinterpret_cast<uintptr_t>(x_bf16) | reinterpret_cast<uintptr_t>(a1_q) |
                        reinterpret_cast<uintptr_t>(a1_sf) | reinterpret_cast<uintptr_t>(x_q);
  if (T > 0 && (mis & 15u) != 0)
    return fail(NVFP4_ERR_ALIGNMENT, "moe_route_permute_static: x, a1_q and a1_sf must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(x_global_scale) & 3u) != 0)
    return fail(NVFP4_ERR_ALIGNMENT, "moe_route_permute_static: x_global_scale not 4-byte aligned");
  const size_t need = moe_route_permute_workspace(T, H, E, top_k);
  if (need > kStaticScratchBytes)
    return fail(NVFP4_ERR_UNSUPPORTED,
                "moe_route_permute_static: needs %zu bytes of scratch, more than its fixed %zu-byte device array "
                "(use moe_route_permute with a workspace)",
                need, kStaticScratchBytes);
  uint8_t* ws = nullptr;
  nvfp4_status st = static_scratch(&ws);
  if (st != NVFP4_OK) return st;

  RouteBuffers b;
  b.logits = logits;
  b.x = x_bf16;
  b.T = T;
  b.H = H;
  b.E = E;
  b.top_k = top_k;
  b.topk_ids = topk_ids;
  b.topk_w = topk_w;
  b.counts = expert_counts;
  b.offsets = expert_offsets;
  b.perm_token = perm_token;
  b.inv_perm = inv_perm;
  b.a1_q = a1_q;
  b.a1_sf = a1_sf;
  b.x_q = x_q;
  b.x_gscale = x_global_scale;
  b.rows_max = moe_padded_rows_max(T, E, top_k);
  route_carve_workspace(b, ws);
  cudaError_t e = route_permute_launch(b, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : fail_cuda(e, "moe_route_permute_static");
}

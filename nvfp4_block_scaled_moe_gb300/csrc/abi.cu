// The extern "C" boundary of libnvfp4moe.so: argument checks (before any CUDA
// call), status codes, thread-local error messages, the per-device error word
// and the bounded-wait self-test.  Compute lives in quantize.cu, route.cu and
// gemm.cu.
#include <stdarg.h>
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

__device__ unsigned g_error_word;

static thread_local char g_msg[512] = "";

nvfp4_status fail(nvfp4_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

nvfp4_status fail_cuda(cudaError_t e, const char* where) {
  return fail(NVFP4_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

unsigned* device_error_word() {
  static unsigned* addr[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) == cudaSuccess) addr[dev] = static_cast<unsigned*>(p);
  }
  return addr[dev];
}

__global__ void selftest_wait_kernel(const volatile int32_t* flag, int64_t limit_ns, unsigned* err) {
  if (threadIdx.x != 0) return;
  const uint64_t t0 = globaltimer_ns();
  while (*flag == 0) {
    if (globaltimer_ns() - t0 > static_cast<uint64_t>(limit_ns)) {
      raise_error(err, kErrTimeout);
      return;
    }
  }
}

cudaError_t selftest_wait_launch(const int32_t* flag, int64_t limit_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(flag, limit_ns, device_error_word());
  return cudaGetLastError();
}

static bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace nvfp4

using namespace nvfp4;

#define CHECK_ARG(cond, ...)                                         \
  do {                                                               \
    if (!(cond)) return fail(NVFP4_ERR_INVALID_ARG, __VA_ARGS__);   \
  } while (0)
#define CHECK_SUP(cond, ...)                                         \
  do {                                                               \
    if (!(cond)) return fail(NVFP4_ERR_UNSUPPORTED, __VA_ARGS__);   \
  } while (0)
#define CHECK_AL(cond, ...)                                          \
  do {                                                               \
    if (!(cond)) return fail(NVFP4_ERR_ALIGNMENT, __VA_ARGS__);     \
  } while (0)

extern "C" {

size_t nvfp4_sf_bytes(int64_t rows, int64_t cols) {
  if (rows <= 0 || cols <= 0) return 0;
  return static_cast<size_t>((rows + 127) / 128) * static_cast<size_t>((cols + 63) / 64) * 512u;
}

int64_t moe_padded_rows_max(int32_t T, int32_t E, int32_t top_k) {
  if (T <= 0 || E <= 0 || top_k <= 0) return 0;
  const int64_t routed = static_cast<int64_t>(T) * top_k;
  const int64_t groups = routed < E ? routed : E;
  return ((routed + 127 * groups) / 128) * 128;
}

size_t moe_route_permute_workspace(int32_t T, int32_t H, int32_t E, int32_t top_k) {
  (void)top_k;
  if (T < 0 || H <= 0 || E <= 0) return 0;
  return route_workspace_bytes(T, E);
}

const char* nvfp4_last_error(void) { return g_msg; }

nvfp4_status nvfp4_quantize(const void* in, nvfp4_in_dtype dtype, nvfp4_quant_mode mode, int64_t rows,
                            int64_t out_cols, int64_t in_ld_elems, uint8_t* q_out, uint8_t* sf_out,
                            const float* global_scale, float* h_debug, nvfp4_stream_t stream) {
  CHECK_ARG(in && q_out && sf_out, "nvfp4_quantize: null pointer");
  CHECK_ARG(dtype == NVFP4_IN_BF16 || dtype == NVFP4_IN_F32, "nvfp4_quantize: bad dtype %d", (int)dtype);
  CHECK_ARG(mode == NVFP4_MODE_PLAIN || mode == NVFP4_MODE_SWIGLU_GU8 || mode == NVFP4_MODE_DEINTERLEAVE_GU8,
            "nvfp4_quantize: bad mode %d", (int)mode);
  CHECK_ARG(rows > 0 && out_cols > 0, "nvfp4_quantize: rows and out_cols must be positive");
  CHECK_SUP(out_cols % 16 == 0, "nvfp4_quantize: out_cols=%lld is not a multiple of 16", (long long)out_cols);
  CHECK_SUP(mode == NVFP4_MODE_PLAIN || dtype == NVFP4_IN_BF16, "nvfp4_quantize: the GU8 modes take BF16 input");
  const int64_t in_cols = mode == NVFP4_MODE_PLAIN ? out_cols : 2 * out_cols;
  CHECK_ARG(in_ld_elems >= in_cols, "nvfp4_quantize: in_ld_elems=%lld < %lld", (long long)in_ld_elems,
            (long long)in_cols);
  const int64_t esize = dtype == NVFP4_IN_BF16 ? 2 : 4;
  CHECK_AL(al16(in) && (in_ld_elems * esize) % 16 == 0, "nvfp4_quantize: input not 16-byte aligned");
  // a 16-block's eight nibble bytes leave as one 8-byte store, a row's four scales as one word
  CHECK_AL((reinterpret_cast<uintptr_t>(q_out) & 7u) == 0 && (reinterpret_cast<uintptr_t>(sf_out) & 3u) == 0,
           "nvfp4_quantize: q_out must be 8-byte and sf_out 4-byte aligned");
  CHECK_AL(h_debug == nullptr || al16(h_debug), "nvfp4_quantize: h_debug not 16-byte aligned");
  CHECK_AL(al4(global_scale), "nvfp4_quantize: global_scale not 4-byte aligned");
  cudaError_t e = quantize_launch(in, dtype, mode, rows, out_cols, in_ld_elems, q_out, sf_out, 0, global_scale,
                                  h_debug, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : fail_cuda(e, "nvfp4_quantize");
}

nvfp4_status nvfp4_global_scale(const void* in, nvfp4_in_dtype dtype, int64_t rows, int64_t cols,
                                int64_t in_ld_elems, float* g_out, nvfp4_stream_t stream) {
  CHECK_ARG(in && g_out, "nvfp4_global_scale: null pointer");
  CHECK_ARG(dtype == NVFP4_IN_BF16 || dtype == NVFP4_IN_F32, "nvfp4_global_scale: bad dtype %d", (int)dtype);
  CHECK_ARG(rows > 0 && cols > 0, "nvfp4_global_scale: rows and cols must be positive");
  CHECK_SUP(cols % 8 == 0, "nvfp4_global_scale: cols=%lld is not a multiple of 8", (long long)cols);
  CHECK_ARG(in_ld_elems >= cols, "nvfp4_global_scale: in_ld_elems=%lld < cols", (long long)in_ld_elems);
  const int64_t esize = dtype == NVFP4_IN_BF16 ? 2 : 4;
  CHECK_AL(al16(in) && (in_ld_elems * esize) % 16 == 0, "nvfp4_global_scale: input not 16-byte aligned");
  CHECK_AL(al4(g_out), "nvfp4_global_scale: g_out not 4-byte aligned");
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail_cuda(e, "nvfp4_global_scale: device query");
  e = global_scale_launch(in, dtype, rows, cols, in_ld_elems, g_out, sms, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : fail_cuda(e, "nvfp4_global_scale");
}

nvfp4_status nvfp4_sf_swizzle(const uint8_t* sf_in, int64_t mn_rows, int64_t k_sf_cols, int64_t stride_mn,
                              int64_t stride_ksf, uint8_t* sf_out, int inverse, nvfp4_stream_t stream) {
  CHECK_ARG(sf_in && sf_out, "nvfp4_sf_swizzle: null pointer");
  CHECK_ARG(mn_rows > 0 && k_sf_cols > 0, "nvfp4_sf_swizzle: sizes must be positive");
  CHECK_ARG(stride_mn > 0 && stride_ksf > 0, "nvfp4_sf_swizzle: strides must be positive");
  CHECK_AL(inverse || (reinterpret_cast<uintptr_t>(sf_out) & 3u) == 0,
           "nvfp4_sf_swizzle: swizzled output must be 4-byte aligned");
  cudaError_t e = sf_swizzle_launch(sf_in, mn_rows, k_sf_cols, stride_mn, stride_ksf, sf_out, inverse,
                                    reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : fail_cuda(e, "nvfp4_sf_swizzle");
}

nvfp4_status moe_route_permute(const float* logits, const void* x_bf16, int32_t T, int32_t H, int32_t E,
                               int32_t top_k, int32_t* topk_ids, float* topk_w, int32_t* expert_counts,
                               int32_t* expert_offsets, int32_t* perm_token, int32_t* inv_perm, uint8_t* a1_q,
                               uint8_t* a1_sf, uint8_t* x_q, const float* x_global_scale, void* workspace,
                               size_t workspace_bytes, nvfp4_stream_t stream) {
  CHECK_ARG(T >= 0, "moe_route_permute: T=%d", T);
  CHECK_ARG(expert_counts && expert_offsets && workspace, "moe_route_permute: null pointer");
  CHECK_ARG(T == 0 || (logits && topk_ids && topk_w && perm_token && inv_perm), "moe_route_permute: null pointer");
  // a1_sf NULL: routing only (a1_q and x_q NULL too); else x and a1_q and / or x_q
  CHECK_ARG(T == 0 || (a1_sf ? (x_bf16 && (a1_q || x_q)) : (!a1_q && !x_q)),
            "moe_route_permute: staging needs x, a1_sf and a1_q or x_q (routing only: all four NULL)");
  CHECK_SUP(E >= 1 && E <= 1024, "moe_route_permute: E=%d outside [1, 1024]", E);
  CHECK_SUP(top_k >= 1 && top_k <= E && top_k <= 32, "moe_route_permute: top_k=%d outside [1, min(E, 32)]", top_k);
  CHECK_SUP(H > 0 && H % 64 == 0, "moe_route_permute: H=%d is not a positive multiple of 64", H);
  CHECK_AL(al16(workspace) && (T == 0 || (al16(x_bf16) && al16(a1_q) && al16(a1_sf) && al16(x_q))),
           "moe_route_permute: x, a1_q, a1_sf and workspace must be 16-byte aligned");
  CHECK_AL(al4(x_global_scale), "moe_route_permute: x_global_scale not 4-byte aligned");
  const size_t need = moe_route_permute_workspace(T, H, E, top_k);
  CHECK_ARG(workspace_bytes >= need, "moe_route_permute: workspace %zu < %zu bytes", workspace_bytes, need);
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
  route_carve_workspace(b, workspace);
  cudaError_t e = route_permute_launch(b, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : fail_cuda(e, "moe_route_permute");
}

}  // extern "C"

namespace {

// nvfp4_grouped_gemm's argument checks (status and message; nothing launched)
nvfp4_status check_grouped_gemm(const uint8_t* a_q, const uint8_t* a_sf, int64_t rows_max,
                                const int32_t* group_offsets, const int32_t* group_counts, int32_t G, int32_t N,
                                int32_t K, const uint8_t* b_q, const uint8_t* b_sf, const float* a_global_scale,
                                const float* b_global_scale, const float* out_global_scale, nvfp4_epilogue epilogue,
                                uint8_t* out_q, uint8_t* out_sf, void* out_bf16, float* h_debug,
                                const int32_t* a_gather, int64_t a_gather_rows) {
  CHECK_ARG(a_q && a_sf && b_q && b_sf, "nvfp4_grouped_gemm: null operand");
  CHECK_ARG(!a_gather || (a_gather_rows > 0 && a_gather_rows < (int64_t(1) << 31)),
            "nvfp4_grouped_gemm: a_gather_rows=%lld", (long long)a_gather_rows);
  CHECK_AL(al16(a_gather), "nvfp4_grouped_gemm: a_gather not 16-byte aligned");
  CHECK_SUP(!a_gather || epilogue == NVFP4_EPI_SWIGLU_NVFP4,
            "nvfp4_grouped_gemm: gathered A rows are supported with the SwiGLU + NVFP4 epilogue (L1)");
  CHECK_ARG(epilogue == NVFP4_EPI_SWIGLU_NVFP4 || epilogue == NVFP4_EPI_BF16 || epilogue == NVFP4_EPI_SWIGLU_BF16,
            "nvfp4_grouped_gemm: bad epilogue");
  CHECK_ARG(epilogue != NVFP4_EPI_SWIGLU_NVFP4 || (out_q && out_sf), "nvfp4_grouped_gemm: null NVFP4 output");
  CHECK_ARG(epilogue == NVFP4_EPI_SWIGLU_NVFP4 || out_bf16, "nvfp4_grouped_gemm: null BF16 output");
  CHECK_ARG(group_offsets || !group_counts, "nvfp4_grouped_gemm: group_counts needs group_offsets");
  CHECK_ARG(G >= 1 && N > 0 && K > 0 && rows_max > 0, "nvfp4_grouped_gemm: sizes must be positive");
  CHECK_SUP(group_offsets || G == 1, "nvfp4_grouped_gemm: NULL group_offsets means G == 1");
  CHECK_SUP(K % 256 == 0, "nvfp4_grouped_gemm: K=%d is not a multiple of 256", K);
  CHECK_SUP(N % (epilogue == NVFP4_EPI_BF16 ? 128 : 256) == 0,
            "nvfp4_grouped_gemm: N=%d is not a multiple of %d", N, epilogue == NVFP4_EPI_BF16 ? 128 : 256);
  CHECK_SUP(rows_max % 128 == 0 && rows_max < (int64_t(1) << 31), "nvfp4_grouped_gemm: rows_max=%lld",
            (long long)rows_max);
  CHECK_SUP(static_cast<int64_t>(G) * N < (int64_t(1) << 31), "nvfp4_grouped_gemm: G*N too large");
  CHECK_AL(al16(a_q) && al16(a_sf) && al16(b_q) && al16(b_sf), "nvfp4_grouped_gemm: operands not 16-byte aligned");
  CHECK_AL((!out_q || al16(out_q)) && (!out_sf || al16(out_sf)) && (!out_bf16 || al16(out_bf16)) &&
               (!h_debug || al16(h_debug)),
           "nvfp4_grouped_gemm: outputs not 16-byte aligned");
  CHECK_AL(al4(a_global_scale) && al4(b_global_scale) && al4(out_global_scale),
           "nvfp4_grouped_gemm: global scales not 4-byte aligned");
  return NVFP4_OK;
}

// a side combine job's checks (moe_combine's, without shared rows)
nvfp4_status check_combine_job(const nvfp4_combine_job* c) {
  if (c == nullptr) return NVFP4_OK;
  CHECK_ARG(c->T >= 0 && c->top_k >= 1 && c->top_k <= 32, "combine job: T=%d top_k=%d", c->T, c->top_k);
  if (c->T == 0) return NVFP4_OK;
  CHECK_ARG(c->rows_bf16 && c->inv_perm && c->topk_w && c->y_bf16, "combine job: null pointer");
  CHECK_ARG(c->rows >= 1, "combine job: rows=%lld", (long long)c->rows);
  CHECK_SUP(c->H > 0 && c->H % 8 == 0, "combine job: H=%d is not a positive multiple of 8", c->H);
  CHECK_AL(al16(c->rows_bf16) && al16(c->y_bf16), "combine job: rows and y must be 16-byte aligned");
  return NVFP4_OK;
}

// a staging job's checks (moe_route_permute's, for the staging half)
nvfp4_status check_stage_job(const nvfp4_stage_job* j) {
  if (j == nullptr) return NVFP4_OK;
  CHECK_ARG(j->T >= 0, "stage job: T=%d", j->T);
  if (j->T == 0) return NVFP4_OK;
  CHECK_ARG(j->x_bf16 && j->inv_perm && j->expert_counts && j->expert_offsets && j->a1_q && j->a1_sf,
            "stage job: null pointer");
  CHECK_SUP(j->E >= 1 && j->E <= 1024, "stage job: E=%d outside [1, 1024]", j->E);
  CHECK_SUP(j->top_k >= 1 && j->top_k <= j->E && j->top_k <= 32, "stage job: top_k=%d outside [1, min(E, 32)]",
            j->top_k);
  CHECK_SUP(j->H > 0 && j->H % 64 == 0, "stage job: H=%d is not a positive multiple of 64", j->H);
  CHECK_SUP(j->rows_max > 0 && j->rows_max % 128 == 0 && j->rows_max < (int64_t(1) << 31),
            "stage job: rows_max=%lld is not a positive multiple of 128", (long long)j->rows_max);
  CHECK_AL(al16(j->x_bf16) && al16(j->a1_q) && al16(j->a1_sf), "stage job: x, a1_q and a1_sf must be 16-byte aligned");
  CHECK_AL(al4(j->x_global_scale), "stage job: x_global_scale not 4-byte aligned");
  return NVFP4_OK;
}

StageJob stage_job(const nvfp4_stage_job& j) {
  StageJob s;
  s.x = j.x_bf16;
  s.x_gscale = j.x_global_scale;
  s.inv_perm = j.inv_perm;
  s.counts = j.expert_counts;
  s.offsets = j.expert_offsets;
  s.a_q = j.a1_q;
  s.a_sf = j.a1_sf;
  s.x_q = nullptr;
  s.T = j.T;
  s.H = j.H;
  s.E = j.E;
  s.k = j.top_k;
  s.rows_max = j.rows_max;
  s.err = device_error_word();
  return s;
}

GemmArgs make_gemm_args(const uint8_t* a_q, const uint8_t* a_sf, int64_t rows_max, const int32_t* group_offsets,
                        const int32_t* group_counts, int32_t G, int32_t N, int32_t K, const uint8_t* b_q,
                        const uint8_t* b_sf, float alpha, const float* a_global_scale, const float* b_global_scale,
                        const float* out_global_scale, nvfp4_epilogue epilogue, uint8_t* out_q, uint8_t* out_sf,
                        void* out_bf16, float* h_debug, const int32_t* a_gather, int64_t a_gather_rows) {
  GemmArgs a;
  a.a_q = a_q;
  a.a_sf = a_sf;
  a.rows_max = rows_max;
  a.a_gather = a_gather;
  a.a_rows = a_gather ? a_gather_rows : rows_max;
  a.offsets = group_offsets;
  a.counts = group_counts;
  a.G = G;
  a.N = N;
  a.K = K;
  a.b_q = b_q;
  a.b_sf = b_sf;
  a.alpha = alpha;
  a.a_gscale = a_global_scale;
  a.b_gscale = b_global_scale;
  a.out_gscale = out_global_scale;
  a.epilogue = epilogue;
  a.out_q = out_q;
  a.out_sf = out_sf;
  a.out_bf16 = out_bf16;
  a.h_debug = h_debug;
  return a;
}

}  // namespace

extern "C" {

nvfp4_status nvfp4_grouped_gemm(const uint8_t* a_q, const uint8_t* a_sf, int64_t rows_max,
                                const int32_t* group_offsets, const int32_t* group_counts, int32_t G, int32_t N,
                                int32_t K, const uint8_t* b_q, const uint8_t* b_sf, float alpha,
                                const float* a_global_scale, const float* b_global_scale,
                                const float* out_global_scale, nvfp4_epilogue epilogue, uint8_t* out_q,
                                uint8_t* out_sf, void* out_bf16, float* h_debug, const int32_t* a_gather,
                                int64_t a_gather_rows, const nvfp4_combine_job* side_combine,
                                const nvfp4_stage_job* side_stage, nvfp4_stream_t stream) {
  nvfp4_status st = check_combine_job(side_combine);
  if (st == NVFP4_OK) st = check_stage_job(side_stage);
  if (st != NVFP4_OK) return st;
  st = check_grouped_gemm(a_q, a_sf, rows_max, group_offsets, group_counts, G, N, K, b_q, b_sf, a_global_scale,
                         b_global_scale, out_global_scale, epilogue, out_q, out_sf, out_bf16, h_debug, a_gather,
                         a_gather_rows);
  if (st != NVFP4_OK) return st;
  GemmArgs a = make_gemm_args(a_q, a_sf, rows_max, group_offsets, group_counts, G, N, K, b_q, b_sf, alpha,
                              a_global_scale, b_global_scale, out_global_scale, epilogue, out_q, out_sf, out_bf16,
                              h_debug, a_gather, a_gather_rows);
  if (side_combine != nullptr && side_combine->T > 0) {
    a.side_rows = side_combine->rows_bf16;
    a.side_n_rows = side_combine->rows;
    a.side_inv = side_combine->inv_perm;
    a.side_w = side_combine->topk_w;
    a.side_y = side_combine->y_bf16;
    a.side_T = side_combine->T;
    a.side_H = side_combine->H;
    a.side_k = side_combine->top_k;
  }
  if (side_stage != nullptr && side_stage->T > 0) a.stage = stage_job(*side_stage);
  return gemm_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

nvfp4_status moe_stage_activation(const nvfp4_stage_job* job, nvfp4_stream_t stream) {
  CHECK_ARG(job != nullptr, "moe_stage_activation: null job");
  const nvfp4_status st = check_stage_job(job);
  if (st != NVFP4_OK) return st;
  const cudaError_t e = stage_launch(stage_job(*job), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : fail_cuda(e, "moe_stage_activation");
}

nvfp4_status nvfp4_moe_ffn_forward(const uint8_t* a1_q, const uint8_t* a1_sf, const int32_t* expert_offsets,
                                   const int32_t* expert_counts, int32_t E, int32_t H, int32_t I, int64_t rows_max,
                                   const uint8_t* w1_q, const uint8_t* w1_sf, const uint8_t* w2_q,
                                   const uint8_t* w2_sf, float alpha1, float alpha2, const float* x_global_scale,
                                   const float* w1_global_scale, const float* a2_global_scale,
                                   const float* w2_global_scale, uint8_t* a2_q, uint8_t* a2_sf, void* rows_out_bf16,
                                   float* h_debug, const int32_t* a1_gather, int64_t a1_gather_rows,
                                   const nvfp4_combine_job* prev_combine, nvfp4_stream_t stream) {
  CHECK_ARG(expert_offsets && expert_counts, "nvfp4_moe_ffn_forward: null expert offsets/counts");
  CHECK_ARG(prev_combine == nullptr || prev_combine->T == 0 || prev_combine->H == H,
            "nvfp4_moe_ffn_forward: prev_combine H=%d differs from H=%d", prev_combine ? prev_combine->H : 0, H);
  CHECK_ARG(a2_q && a2_sf && rows_out_bf16, "nvfp4_moe_ffn_forward: null output");
  CHECK_SUP(H > 0 && H % 256 == 0 && I > 0 && I % 256 == 0,
            "nvfp4_moe_ffn_forward: H=%d and I=%d must be positive multiples of 256", H, I);
  nvfp4_status st = nvfp4_grouped_gemm(a1_q, a1_sf, rows_max, expert_offsets, expert_counts, E, 2 * I, H, w1_q,
                                       w1_sf, alpha1, x_global_scale, w1_global_scale, a2_global_scale,
                                       NVFP4_EPI_SWIGLU_NVFP4, a2_q, a2_sf, nullptr, h_debug, a1_gather,
                                       a1_gather_rows, prev_combine, nullptr, stream);
  if (st != NVFP4_OK) return st;
  return nvfp4_grouped_gemm(a2_q, a2_sf, rows_max, expert_offsets, expert_counts, E, H, I, w2_q, w2_sf, alpha2,
                            a2_global_scale, w2_global_scale, nullptr, NVFP4_EPI_BF16, nullptr, nullptr,
                            rows_out_bf16, nullptr, nullptr, 0, nullptr, nullptr, stream);
}

nvfp4_status moe_combine(const void* rows_bf16, const int32_t* inv_perm, const float* topk_w, int32_t T,
                         int32_t H, int32_t top_k, const void* shared_bf16, void* y_bf16, nvfp4_stream_t stream) {
  CHECK_ARG(T >= 0 && top_k >= 1, "moe_combine: T=%d top_k=%d", T, top_k);
  CHECK_ARG(T == 0 || (rows_bf16 && inv_perm && topk_w && y_bf16), "moe_combine: null pointer");
  CHECK_SUP(H > 0 && H % 8 == 0, "moe_combine: H=%d is not a positive multiple of 8", H);
  CHECK_AL(T == 0 || (al16(rows_bf16) && al16(y_bf16)), "moe_combine: rows and y must be 16-byte aligned");
  CHECK_AL(al16(shared_bf16), "moe_combine: shared rows must be 16-byte aligned");
  // rows_bf16's row count is not an argument: only negative rows are caught
  cudaError_t e = combine_launch(rows_bf16, INT64_MAX, inv_perm, topk_w, T, H, top_k, shared_bf16, y_bf16,
                                 reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : fail_cuda(e, "moe_combine");
}

}  // extern "C"

namespace {

// the checks of buffer set b for a batch of T tokens (device buffers and sizes)
nvfp4_status check_buffers(int32_t T, int32_t H, int32_t I, int32_t E, int32_t top_k, const nvfp4_moe_weights* w,
                           const nvfp4_moe_buffers* b) {
  CHECK_ARG(w && b, "host step: null pointer");
  CHECK_ARG(T >= 1, "host step: T=%d", T);
  CHECK_ARG(b->x_bf16 && b->logits && b->y_bf16 && b->rows_bf16 && b->topk_ids && b->topk_w && b->expert_counts &&
                b->expert_offsets && b->perm_token && b->inv_perm && b->a1_q && b->a1_sf && b->a2_q && b->a2_sf &&
                b->workspace && w->w1_q && w->w1_sf && w->w2_q && w->w2_sf,
            "host step: null device buffer");
  // the checks of the calls, before anything is enqueued
  CHECK_SUP(E >= 1 && E <= 1024, "host step: E=%d outside [1, 1024]", E);
  CHECK_SUP(top_k >= 1 && top_k <= E && top_k <= 32, "host step: top_k=%d", top_k);
  CHECK_SUP(H > 0 && H % 256 == 0 && I > 0 && I % 256 == 0,
            "host step: H=%d and I=%d must be positive multiples of 256", H, I);
  CHECK_ARG(b->rows_max >= moe_padded_rows_max(T, E, top_k), "host step: rows_max=%lld < moe_padded_rows_max",
            (long long)b->rows_max);
  CHECK_ARG(b->workspace_bytes >= moe_route_permute_workspace(T, H, E, top_k), "host step: workspace too small");
  CHECK_AL(al16(b->x_bf16) && al16(b->y_bf16) && al16(b->rows_bf16) && al16(b->a1_q) && al16(b->a1_sf) &&
               al16(b->a2_q) && al16(b->a2_sf) && al16(b->workspace) && al16(w->w1_q) && al16(w->w1_sf) &&
               al16(w->w2_q) && al16(w->w2_sf),
           "host step: device buffers must be 16-byte aligned");
  CHECK_SUP(b->rows_max % 128 == 0 && b->rows_max < (int64_t(1) << 31), "host step: rows_max=%lld",
            (long long)b->rows_max);
  return NVFP4_OK;
}

// host x and logits -> b's device x and logits, then an optional wait
nvfp4_status enqueue_copy_in(const void* x_host, const float* logits_host, int32_t T, int32_t H, int32_t E,
                             const nvfp4_moe_buffers* b, cudaEvent_t compute_after, cudaStream_t s) {
  cudaError_t e = cudaMemcpyAsync(b->x_bf16, x_host, static_cast<size_t>(T) * H * 2, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(b->logits, logits_host, static_cast<size_t>(T) * E * sizeof(float), cudaMemcpyHostToDevice,
                        s);
  if (e == cudaSuccess && compute_after != nullptr) e = cudaStreamWaitEvent(s, compute_after, 0);
  return e == cudaSuccess ? NVFP4_OK : fail_cuda(e, "host step: copy in");
}

// routing of b's batch; staged into a1 unless `stage` is false (routing only)
nvfp4_status enqueue_route(int32_t T, int32_t H, int32_t E, int32_t top_k, const nvfp4_moe_buffers* b, bool stage,
                           nvfp4_stream_t stream) {
  return moe_route_permute(b->logits, b->x_bf16, T, H, E, top_k, b->topk_ids, b->topk_w, b->expert_counts,
                           b->expert_offsets, b->perm_token, b->inv_perm, stage ? b->a1_q : nullptr,
                           stage ? b->a1_sf : nullptr, nullptr, nullptr, b->workspace, b->workspace_bytes, stream);
}

nvfp4_status enqueue_l1(int32_t H, int32_t I, int32_t E, const nvfp4_moe_weights* w, const nvfp4_moe_buffers* b,
                        const nvfp4_combine_job* side, nvfp4_stream_t stream) {
  return nvfp4_grouped_gemm(b->a1_q, b->a1_sf, b->rows_max, b->expert_offsets, b->expert_counts, E, 2 * I, H,
                            w->w1_q, w->w1_sf, 1.0f, nullptr, nullptr, nullptr, NVFP4_EPI_SWIGLU_NVFP4, b->a2_q,
                            b->a2_sf, nullptr, nullptr, nullptr, 0, side, nullptr, stream);
}

nvfp4_status enqueue_l2(int32_t H, int32_t I, int32_t E, const nvfp4_moe_weights* w, const nvfp4_moe_buffers* b,
                        const nvfp4_stage_job* side, nvfp4_stream_t stream) {
  return nvfp4_grouped_gemm(b->a2_q, b->a2_sf, b->rows_max, b->expert_offsets, b->expert_counts, E, H, I, w->w2_q,
                            w->w2_sf, 1.0f, nullptr, nullptr, nullptr, NVFP4_EPI_BF16, nullptr, nullptr,
                            b->rows_bf16, nullptr, nullptr, 0, nullptr, side, stream);
}

nvfp4_status copy_out(const nvfp4_moe_buffers* b, int32_t T, int32_t H, void* y_host, cudaStream_t s,
                      const char* where) {
  const cudaError_t e = cudaMemcpyAsync(y_host, b->y_bf16, static_cast<size_t>(T) * H * 2, cudaMemcpyDeviceToHost, s);
  return e == cudaSuccess ? NVFP4_OK : fail_cuda(e, where);
}

}  // namespace

extern "C" {

nvfp4_status nvfp4_moe_forward_host(const void* x_host, const float* logits_host, void* y_host, int32_t T,
                                    int32_t H, int32_t I, int32_t E, int32_t top_k, const nvfp4_moe_weights* w,
                                    const nvfp4_moe_buffers* b, nvfp4_stream_t stream) {
  CHECK_ARG(x_host && logits_host && y_host, "nvfp4_moe_forward_host: null host pointer");
  nvfp4_status st = check_buffers(T, H, I, E, top_k, w, b);
  if (st != NVFP4_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = enqueue_copy_in(x_host, logits_host, T, H, E, b, nullptr, s);
  if (st == NVFP4_OK) st = enqueue_route(T, H, E, top_k, b, true, stream);
  if (st == NVFP4_OK) st = enqueue_l1(H, I, E, w, b, nullptr, stream);
  if (st == NVFP4_OK) st = enqueue_l2(H, I, E, w, b, nullptr, stream);
  if (st == NVFP4_OK) st = moe_combine(b->rows_bf16, b->inv_perm, b->topk_w, T, H, top_k, nullptr, b->y_bf16, stream);
  if (st != NVFP4_OK) return st;
  return copy_out(b, T, H, y_host, s, "nvfp4_moe_forward_host: copy out");
}

nvfp4_status nvfp4_moe_step_host(const void* x_host, const float* logits_host, int32_t T, int32_t H, int32_t I,
                                 int32_t E, int32_t top_k, const nvfp4_moe_weights* w, const nvfp4_moe_buffers* b,
                                 const nvfp4_moe_buffers* prev, int32_t prev_T, void* prev_y_host,
                                 nvfp4_event_t compute_after, nvfp4_event_t compute_done, nvfp4_stream_t stream) {
  CHECK_ARG(x_host && logits_host, "nvfp4_moe_step_host: null host pointer");
  nvfp4_status st = check_buffers(T, H, I, E, top_k, w, b);
  if (st != NVFP4_OK) return st;
  if (prev != nullptr) {
    CHECK_ARG(prev != b, "nvfp4_moe_step_host: prev is this step's buffer set");
    CHECK_ARG(prev_y_host, "nvfp4_moe_step_host: prev needs prev_y_host");
    st = check_buffers(prev_T, H, I, E, top_k, w, prev);
    if (st != NVFP4_OK) return st;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = enqueue_copy_in(x_host, logits_host, T, H, E, b, reinterpret_cast<cudaEvent_t>(compute_after), s);
  if (st != NVFP4_OK) return st;
  if (prev == nullptr) {
    st = enqueue_route(T, H, E, top_k, b, true, stream);
    if (st == NVFP4_OK) st = enqueue_l1(H, I, E, w, b, nullptr, stream);
  } else {
    // routing only; prev's L2 stages this batch on its spare warps; this batch's
    // L1 runs prev's combine on its spare warps
    nvfp4_stage_job stage = {};
    stage.x_bf16 = b->x_bf16;
    stage.inv_perm = b->inv_perm;
    stage.expert_counts = b->expert_counts;
    stage.expert_offsets = b->expert_offsets;
    stage.a1_q = b->a1_q;
    stage.a1_sf = b->a1_sf;
    stage.T = T;
    stage.H = H;
    stage.E = E;
    stage.top_k = top_k;
    stage.rows_max = b->rows_max;
    nvfp4_combine_job comb = {};
    comb.rows_bf16 = prev->rows_bf16;
    comb.inv_perm = prev->inv_perm;
    comb.topk_w = prev->topk_w;
    comb.T = prev_T;
    comb.top_k = top_k;
    comb.H = H;
    comb.y_bf16 = prev->y_bf16;
    comb.rows = prev->rows_max;
    st = enqueue_route(T, H, E, top_k, b, false, stream);
    if (st == NVFP4_OK) st = enqueue_l2(H, I, E, w, prev, &stage, stream);
    if (st == NVFP4_OK) st = enqueue_l1(H, I, E, w, b, &comb, stream);
  }
  if (st != NVFP4_OK) return st;
  if (compute_done != nullptr) {
    const cudaError_t e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(compute_done), s);
    if (e != cudaSuccess) return fail_cuda(e, "nvfp4_moe_step_host: event");
  }
  return prev != nullptr ? copy_out(prev, prev_T, H, prev_y_host, s, "nvfp4_moe_step_host: copy out") : NVFP4_OK;
}

nvfp4_status nvfp4_moe_finish_host(const nvfp4_moe_weights* w, const nvfp4_moe_buffers* b, int32_t T, int32_t H,
                                   int32_t I, int32_t E, int32_t top_k, void* y_host, nvfp4_stream_t stream) {
  CHECK_ARG(y_host, "nvfp4_moe_finish_host: null y_host");
  nvfp4_status st = check_buffers(T, H, I, E, top_k, w, b);
  if (st == NVFP4_OK) st = enqueue_l2(H, I, E, w, b, nullptr, stream);
  if (st == NVFP4_OK) st = moe_combine(b->rows_bf16, b->inv_perm, b->topk_w, T, H, top_k, nullptr, b->y_bf16, stream);
  if (st != NVFP4_OK) return st;
  return copy_out(b, T, H, y_host, reinterpret_cast<cudaStream_t>(stream), "nvfp4_moe_finish_host: copy out");
}

nvfp4_status nvfp4_device_status(nvfp4_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "nvfp4_device_status: stream");
  unsigned word = 0;
  e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word));
  if (e != cudaSuccess) return fail_cuda(e, "nvfp4_device_status: read");
  if (word == 0) return NVFP4_OK;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
  if (e != cudaSuccess) return fail_cuda(e, "nvfp4_device_status: clear");
  if (word & kErrTimeout) return fail(NVFP4_ERR_TIMEOUT, "device: a bounded wait timed out (word 0x%x)", word);
  return fail(NVFP4_ERR_DEVICE, "device: an index check failed (word 0x%x)", word);
}

nvfp4_status nvfp4_set_gemm_tiles(int32_t mode) { return set_gemm_tiles(mode); }

nvfp4_status nvfp4_selftest_bounded_wait(const int32_t* flag, int64_t limit_ns, nvfp4_stream_t stream) {
  CHECK_ARG(flag != nullptr, "nvfp4_selftest_bounded_wait: null flag");
  CHECK_ARG(limit_ns > 0 && limit_ns <= 10000000000ll, "nvfp4_selftest_bounded_wait: limit_ns outside (0, 10 s]");
  cudaError_t e = selftest_wait_launch(flag, limit_ns, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NVFP4_OK : fail_cuda(e, "nvfp4_selftest_bounded_wait");
}

}  // extern "C"

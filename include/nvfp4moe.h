/*
 * nvfp4moe.h -- C ABI of libnvfp4moe.so, the NVFP4 mixture-of-experts expert FFN
 * for GB300 (sm_103a).
 *
 * The path (the "NVFP4 MegaMoE Debug Log", section "NVFP4 MoE Pipeline"):
 *   moe_route_permute      top-k routing, 128-padded expert grouping, and the
 *                          activation staged to NVFP4 in permuted row order
 *                          (the staging alone: moe_stage_activation)
 *   nvfp4_moe_ffn_forward  L1 block-scaled grouped GEMM -> fused SwiGLU + NVFP4
 *                          re-quantisation -> L2 block-scaled grouped GEMM
 *   moe_combine            routing-weighted sum of each token's expert rows
 * plus the building blocks nvfp4_quantize, nvfp4_sf_swizzle and
 * nvfp4_grouped_gemm.
 *
 * Number formats (the "NVFP4-1.1 Approach, Part 2" notes):
 *   - E2M1 values, two per byte, element 2i in the low nibble of byte i;
 *   - one FP8 E4M3 scale (bias 7, max 448, no NaN emitted) per 16 consecutive
 *     K elements: scale = E4M3_rne_satfinite(fp32(amax / 6)), values divided by
 *     the decoded scale in fp32, then hs = rne(2 * min(|s|, 6)) and hs/2 snapped
 *     to the E2M1 grid with ties to even (so s = 5.25 -> nibble 6);
 *   - "swizzled" SF layout: the K-major atom of the Debug Log's "CUTLASS SF
 *     Layout" -- 512-byte atoms of 128 rows x 4 scales, byte offset
 *       ((mn/128) * ceil(K/64) + k_sf/4) * 512 + (mn%32)*16 + ((mn/32)%4)*4 + k_sf%4
 *     with buffer size nvfp4_sf_bytes(rows, K) (the "Allocation" section's
 *     size(filter_zeros(layout))); padding bytes are written as zero.
 *
 * Conventions for every call:
 *   - Pointers named *_q, *_sf, rows*, y*, logits, x*, w*, topk_*, expert_*,
 *     perm_*, inv_perm, workspace are DEVICE pointers owned by the caller; the
 *     library never allocates or frees device memory and keeps no state between
 *     calls apart from a per-device error word (a __device__ variable).
 *   - All calls are asynchronous on `stream` (NULL = legacy default stream) and
 *     never synchronise the host, except nvfp4_device_status.
 *   - Host-side argument checks run before any CUDA call; on failure the call
 *     returns the status, launches nothing and records a message that
 *     nvfp4_last_error() returns (thread-local).
 *   - Device-side problems (a bounded wait that timed out, an index out of range)
 *     set bits in the per-device error word; nvfp4_device_status() reports them.
 *   - Tensor-core kernels require an sm_100-family GPU (built for sm_103a).
 */
#ifndef NVFP4MOE_H
#define NVFP4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* nvfp4_stream_t;   /* identical to cudaStream_t */

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad enum */
  NVFP4_ERR_UNSUPPORTED = 2,   /* a size outside what the kernels handle */
  NVFP4_ERR_ALIGNMENT = 3,     /* a pointer or leading dimension not 16-byte aligned */
  NVFP4_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
  NVFP4_ERR_TIMEOUT = 5,       /* a device-side bounded wait gave up */
  NVFP4_ERR_DEVICE = 6         /* a device-side index check failed */
} nvfp4_status;

typedef enum { NVFP4_IN_BF16 = 0, NVFP4_IN_F32 = 1 } nvfp4_in_dtype;

typedef enum {
  NVFP4_MODE_PLAIN = 0,        /* quantise the input values themselves */
  NVFP4_MODE_SWIGLU_GU8 = 1,   /* input holds gate/up columns interleaved 8|8;
                                  quantise h = silu(g) * u */
  NVFP4_MODE_DEINTERLEAVE_GU8 = 2 /* input interleaved 8|8 as above; quantise the
                                  second 8 of every 16 columns as they are (the
                                  pages' deinterleave + quantise of an L1 output
                                  whose up slots already hold SwiGLU values) */
} nvfp4_quant_mode;

typedef enum {
  NVFP4_EPI_SWIGLU_NVFP4 = 0,  /* SwiGLU on interleaved 8|8 columns, then NVFP4 */
  NVFP4_EPI_BF16 = 1,          /* alpha * acc rounded to BF16 */
  NVFP4_EPI_SWIGLU_BF16 = 2    /* SwiGLU on interleaved 8|8 columns, written as compact
                                  BF16 [rows_max, N/2] (the pages' compact SwiGLU
                                  output; no re-quantisation) */
} nvfp4_epilogue;

/* Output-tile kernels of nvfp4_grouped_gemm (see nvfp4_set_gemm_tiles). */
typedef enum {
  NVFP4_GEMM_TILES_AUTO = 0,   /* by shape: CTA pairs when groups average >= 256 rows; with
                                  more than one group, split (see nvfp4_grouped_gemm) */
  NVFP4_GEMM_TILES_SINGLE = 1, /* one CTA per 128-row tile */
  NVFP4_GEMM_TILES_PAIR = 2    /* two CTAs (a cluster) per 256-row tile, where N % 256 == 0
                                  and G <= 512; never split */
} nvfp4_gemm_tiles;

/* Bytes of a swizzled SF buffer for a rows x cols matrix (cols in elements):
 * ceil(rows/128) * ceil(cols/64) * 512.  Returns 0 for non-positive sizes. */
size_t nvfp4_sf_bytes(int64_t rows, int64_t cols);

/* Rows to allocate for the permuted, 128-padded activation of T tokens routed
 * top-k over E experts: the largest possible sum over experts of
 * ceil(count_e / 128) * 128.  A multiple of 128. */
int64_t moe_padded_rows_max(int32_t T, int32_t E, int32_t top_k);

/* Bytes of device workspace moe_route_permute needs. */
size_t moe_route_permute_workspace(int32_t T, int32_t H, int32_t E, int32_t top_k);

/* A combine left over from an earlier batch: moe_combine's arguments without
 * shared rows, y = bf16( sum_j w[t, j] * rows[inv_perm[t, j], :] ).  The
 * CTA-pair L1 GEMM (the SwiGLU + NVFP4 epilogue) can run it on two spare warps
 * per CTA while it computes; see nvfp4_grouped_gemm's side_combine. */
typedef struct {
  const void* rows_bf16;       /* BF16 [*, H]: the earlier batch's L2 rows (16-byte aligned) */
  const int32_t* inv_perm;     /* int32 [T, top_k] */
  const float* topk_w;         /* fp32 [T, top_k] */
  int32_t T;                   /* tokens of the earlier batch (0: no job) */
  int32_t top_k;               /* 1 .. 32 */
  int32_t H;                   /* row length, a positive multiple of 8 */
  void* y_bf16;                /* BF16 [T, H], written (16-byte aligned) */
  int64_t rows;                /* rows of rows_bf16 (>= 1): a slot whose inv_perm entry lies outside
                                  [0, rows) reads nothing, adds 0 and sets the device error word */
} nvfp4_combine_job;

/* The activation staging of a routed batch (moe_route_permute's second half,
 * "stage_activation" into the padded per-expert layout): x quantised once per
 * token (per 16 along H, as fp32(x * g) under a two-level scale) and its bytes
 * written into the token's top_k permuted rows of a1_q / a1_sf; every expert's
 * padding rows get zero scales (their nibbles are not written).  The CTA-pair
 * L2 GEMM (the BF16 epilogue) can run it on two spare warps per CTA while it
 * computes; see nvfp4_grouped_gemm's side_stage. */
typedef struct {
  const void* x_bf16;              /* BF16 [T, H] (16-byte aligned) */
  const float* x_global_scale;     /* NULL or x's device encode scale g */
  const int32_t* inv_perm;         /* int32 [T, top_k]: moe_route_permute's */
  const int32_t* expert_counts;    /* int32 [E]: moe_route_permute's */
  const int32_t* expert_offsets;   /* int32 [E+1]: moe_route_permute's */
  uint8_t* a1_q;                   /* [R_max, H/2], written (16-byte aligned) */
  uint8_t* a1_sf;                  /* nvfp4_sf_bytes(R_max, H), swizzled, written (16-byte aligned) */
  int32_t T;                       /* tokens (0: no job) */
  int32_t H;                       /* a positive multiple of 64 */
  int32_t E;                       /* 1 .. 1024 */
  int32_t top_k;                   /* 1 .. min(E, 32) */
  int64_t rows_max;                /* rows of a1_q (R_max, a positive multiple of 128): a row index, or an
                                      expert's last band, outside it is not written and sets the
                                      device error word */
} nvfp4_stage_job;

/* Two-level scale.  The pages' pipeline carries a per-tensor fp32 global scale
 * beside the per-16 E4M3 scales ("NVFP4 MegaMoE Debug Log", "NVFP4 MoE Pipeline":
 * stage_activation returns an input_global_scale; each GEMM's alpha is
 * igs * global_sf) but prints no formula.  This library's reading: an encode
 * scale g (a device fp32 scalar, or one per expert for weights) multiplies the
 * tensor before the per-16 quantisation, i.e. the quantised values are
 * fp32(v * g); a quantised value decodes as e2m1 * e4m3 / g.  Every argument
 * named *global_scale below is such an encode scale, passed as a device
 * pointer; NULL means g = 1 (the one-level scheme, bit for bit).  The pages' igs
 * and global_sf are the reciprocals 1/g. */

/* ---------------------------------------------------------------------------
 * nvfp4_global_scale -- g = fp32(2688 / amax |in|), the encode scale that puts
 * the tensor's largest magnitude at the top of the E2M1 x E4M3 range (6 x 448);
 * g = 1 when amax is 0 or the quotient is not finite (the dynamic
 * input_global_scale of the pages' stage_activation).
 *   in          rows x cols BF16 or fp32 values, row stride in_ld_elems elements,
 *               16-byte aligned with in_ld_elems * element size a multiple of 16.
 *   cols        a positive multiple of 8.
 *   g_out       device fp32 scalar (written; also used as the reduction's
 *               accumulator, so it must not alias the input).
 * -------------------------------------------------------------------------- */
nvfp4_status nvfp4_global_scale(const void* in, nvfp4_in_dtype dtype, int64_t rows, int64_t cols,
                                int64_t in_ld_elems, float* g_out, nvfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * nvfp4_quantize -- per-16 NVFP4 quantiser ("NVFP4-1.1 Approach, Part 2": the
 * quantize_nvfp4 kernel and the deinterleave + quantise kernel; the E4M3 cast
 * and E2M1 nibble rules above).
 *   in          rows x in_cols values, row stride in_ld_elems elements; in_cols =
 *               out_cols (PLAIN) or 2*out_cols (SWIGLU_GU8 and DEINTERLEAVE_GU8,
 *               BF16 only: columns [g0(8) u0(8) g1(8) u1(8) ...]).  16-byte
 *               aligned, and in_ld_elems * element size a multiple of 16.
 *   out_cols    quantised columns per row, a positive multiple of 16.
 *   q_out       rows x out_cols/2 bytes, row-major (written); 8-byte aligned.
 *   sf_out      nvfp4_sf_bytes(rows, out_cols) bytes, swizzled, 4-byte aligned (every byte written,
 *               padding as zero).
 *   global_scale  NULL or the device fp32 encode scale g (two-level scale): the
 *               quantised values are fp32(h * g).
 *   h_debug     NULL, or rows x out_cols fp32: the values h before g is applied.
 * PLAIN mode is bit-exact against the specification above.  SWIGLU_GU8 computes
 * silu with the fast exponential, so h may differ from a float64 evaluation by
 * a few ulp, which can move a value across a rounding boundary; the codes are
 * bit-exact against the specification applied to the h it reports.
 * -------------------------------------------------------------------------- */
nvfp4_status nvfp4_quantize(const void* in, nvfp4_in_dtype dtype, nvfp4_quant_mode mode,
                            int64_t rows, int64_t out_cols, int64_t in_ld_elems,
                            uint8_t* q_out, uint8_t* sf_out, const float* global_scale,
                            float* h_debug, nvfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * nvfp4_sf_swizzle -- the SF remap of the "NVFP4 MegaMoE Debug Log" ("What the
 * forward mapping does", "Source strides"): for every (mn, k_sf) < (mn_rows, k_sf_cols),
 *   forward (inverse == 0): swz[offset(mn, k_sf)] = lin[mn*stride_mn + k_sf*stride_ksf]
 *   inverse (inverse != 0): lin[mn*stride_mn + k_sf*stride_ksf] = swz[offset(mn, k_sf)]
 * SFA (row-major M x K_sf) uses strides (K_sf, 1); SFB stored K_sf x N uses (1, N).
 * The forward direction writes every byte of the nvfp4_sf_bytes(mn_rows, 16*k_sf_cols)
 * buffer (padding as zero); the inverse writes only the addressed bytes.
 * Strides are in bytes and must be positive.
 * -------------------------------------------------------------------------- */
nvfp4_status nvfp4_sf_swizzle(const uint8_t* sf_in, int64_t mn_rows, int64_t k_sf_cols,
                              int64_t stride_mn, int64_t stride_ksf, uint8_t* sf_out,
                              int inverse, nvfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_route_permute -- routing plus "stage_activation" into the padded
 * per-expert layout ("NVFP4 MegaMoE Debug Log", "NVFP4 MoE Pipeline";
 * "NVFP4-1.1 Approach, Part 2", padded_dst gather / scatter).
 *   logits      fp32 [T, E] router logits.
 *   x_bf16      BF16 [T, H] activations (16-byte aligned).
 *   topk_ids    int32 [T, top_k]: the top_k largest logits per token, in
 *               descending order, ties to the lower expert index.
 *   topk_w      fp32 [T, top_k]: softmax over the selected logits.
 *   expert_counts   int32 [E]: routed rows per expert.
 *   expert_offsets  int32 [E+1]: exclusive prefix sum of ceil(count/128)*128.
 *   perm_token  int32 [R_max] (R_max = moe_padded_rows_max): token of each padded
 *               row; -1 on padding rows inside a group; rows at or past
 *               expert_offsets[E] are not written.  Within an expert, rows are in
 *               ascending token order (deterministic, no atomics in the order).
 *   inv_perm    int32 [T, top_k]: padded row of each (token, slot).
 *   a1_q        [R_max, H/2] NVFP4 rows of x in permuted order.  The nibbles of
 *               padding rows inside groups are not written: their scales are
 *               zero, and a zero scale dequantises every E2M1 code to 0, so a
 *               padding row is an exact zero row of the GEMMs whatever its
 *               nibbles hold.  May be NULL when x_q is given (the permuted copy
 *               is then not written).
 *   a1_sf       nvfp4_sf_bytes(R_max, H) bytes, swizzled; every byte of the
 *               groups' 128-row bands is written, zero on padding rows.
 *               NULL (with a1_q and x_q NULL): routing only -- ids, weights,
 *               counts, offsets, perm_token and inv_perm; the staging then comes
 *               from moe_stage_activation or an L2 GEMM's side_stage.
 *   x_q         NULL, or [T, H/2]: the same NVFP4 rows in token order, for an L1
 *               GEMM that gathers its A rows through perm_token (the
 *               permuted copy of a1_q is then never materialised).
 *   x_global_scale  NULL or x's device encode scale g (the rows hold fp32(x * g)).
 *   workspace   >= moe_route_permute_workspace(T, H, E, top_k) bytes, 16-byte
 *               aligned (per-chunk expert histograms, cleared by the call).
 * Limits: 1 <= E <= 1024, 1 <= top_k <= min(E, 32), H a positive multiple of 64,
 * T >= 0 (T == 0 writes zero offsets and counts).
 * -------------------------------------------------------------------------- */
nvfp4_status moe_route_permute(const float* logits, const void* x_bf16, int32_t T, int32_t H,
                               int32_t E, int32_t top_k, int32_t* topk_ids, float* topk_w,
                               int32_t* expert_counts, int32_t* expert_offsets,
                               int32_t* perm_token, int32_t* inv_perm, uint8_t* a1_q,
                               uint8_t* a1_sf, uint8_t* x_q, const float* x_global_scale,
                               void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_route_permute_static -- moe_route_permute for callers that cannot allocate
 * device memory (an engine that hands out all memory from a pool reserved up
 * front, code under an allocator that must not see extra allocations, or a
 * host path where cudaMalloc, which may synchronise the device, is not
 * allowed).  The source pages have no counterpart of this call.
 *   Arguments and outputs are those of moe_route_permute, without the
 *   workspace: the scratch lives in a fixed 16 MiB device array inside the
 *   library, reserved on every GPU that loads the library until the process
 *   exits.  The call performs no cudaMalloc, cudaFree or other allocation.
 *   Limit: moe_route_permute_workspace(T, H, E, top_k) <= 16 MiB (about 2
 *   million tokens at E = 256); larger problems return NVFP4_ERR_UNSUPPORTED.
 *   All calls on a device share the array and leave its contents behind (each
 *   call clears the part it counts into first); calls that overlap
 *   on the GPU race on the array.  The first call on each device looks up the
 *   array's device address (cudaGetSymbolAddress, with that device current):
 *   make that first call before any stream capture.  The address is kept until
 *   the process exits; do not call this again on a device after cudaDeviceReset.
 * -------------------------------------------------------------------------- */
nvfp4_status moe_route_permute_static(const float* logits, const void* x_bf16, int32_t T, int32_t H,
                                      int32_t E, int32_t top_k, int32_t* topk_ids, float* topk_w,
                                      int32_t* expert_counts, int32_t* expert_offsets,
                                      int32_t* perm_token, int32_t* inv_perm, uint8_t* a1_q,
                                      uint8_t* a1_sf, uint8_t* x_q, const float* x_global_scale,
                                      nvfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_stage_activation -- the staging half of moe_route_permute on its own
 * (see nvfp4_stage_job), for a batch routed with a1_sf NULL.  The bytes it
 * writes equal those of moe_route_permute with staging.
 * Limits and errors: those of moe_route_permute; NVFP4_ERR_INVALID_ARG for a
 * null job or a null pointer in a job with T > 0.
 * -------------------------------------------------------------------------- */
nvfp4_status moe_stage_activation(const nvfp4_stage_job* job, nvfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * nvfp4_grouped_gemm -- block-scaled NVFP4 grouped GEMM on the tcgen05 tensor
 * cores (the L1 "fused_swiglu" and L2 GEMMs of "NVFP4-1.1 Approach, Part 2"):
 *   acc[r, n] = sum_k dq(A)[r, k] * dq(B_g)[n, k] for the group g owning row r,
 * with dq(x) = e2m1(x) * e4m3(scale of x's 16-block).
 *   a_q, a_sf   A: [rows_max, K/2] bytes, SF swizzled for rows_max x K.
 *   group_offsets  device int32 [G+1] row offsets (multiples of 128) or NULL for
 *               one group of rows_max rows.
 *   group_counts   device int32 [G] real rows per group, or NULL: rows of a group
 *               at or past its count are computed but not stored (with NULL
 *               offsets, pass NULL; all rows_max rows are stored).
 *   b_q, b_sf   B: [G, N, K/2] bytes; SF swizzled per group (N x K each,
 *               nvfp4_sf_bytes(N, K) bytes apart).
 *   alpha       fp32 scalar applied to acc.
 *   a_global_scale, b_global_scale  NULL or the two-level encode scales of A
 *               (device scalar) and of each group's B (device fp32 [G]): group g
 *               then applies alpha_g = alpha / (g_A * g_B[g]) (one IEEE quotient
 *               of alpha by the fp32 product) in place of alpha.
 *   out_global_scale  NULL or the encode scale of the SwiGLU output: the
 *               re-quantised values are fp32(h * g) (h_debug keeps h).
 *   a_gather, a_gather_rows  NULL, or device int32 [rows_max] (16-byte aligned):
 *               row r of A is row a_gather[r] of a_q, which then has
 *               a_gather_rows rows (loaded with TMA tile::gather4; moe_route_permute's
 *               perm_token over its x_q).  An entry < 0 marks a row whose scales
 *               in a_sf are zero (group padding) and reads row 0; an entry past
 *               the end reads row 0 and sets the device error word.  a_sf keeps
 *               the rows_max-row layout.  Supported with NVFP4_EPI_SWIGLU_NVFP4
 *               (the L1 GEMM); NVFP4_ERR_UNSUPPORTED otherwise.
 *   side_combine  NULL, or the combine of an EARLIER batch to run alongside
 *               (see nvfp4_combine_job).  Its inputs must be complete when this
 *               call's work starts on `stream`, and its buffers must not
 *               overlap this call's.  With the SwiGLU + NVFP4 epilogue on CTA
 *               pairs, two extra warps per CTA stream it while the GEMM runs:
 *               the GEMM moves little DRAM traffic of its own, so the combine's
 *               HBM time mostly hides.  Otherwise (or when the GEMM has tiles
 *               for fewer than half the SMs) it runs as its own launch first.  Either way y equals moe_combine's bit for bit (the
 *               same fp32 slot-order sum and one rounding).
 *   side_stage  NULL, or the activation staging of a LATER batch to run
 *               alongside (see nvfp4_stage_job), under the same rules: inputs
 *               complete when this call's work starts, buffers disjoint from
 *               this call's.  With the BF16 epilogue on CTA pairs (the L2
 *               GEMM), two extra warps per CTA run it while the GEMM computes;
 *               otherwise (or with tiles for fewer than half the SMs) it runs
 *               as its own launch first.  Either way the
 *               bytes equal moe_stage_activation's.
 *   epilogue    NVFP4_EPI_SWIGLU_NVFP4: N columns interleaved 8|8 as gate/up;
 *               h = silu(alpha*g) * (alpha*u) quantised as in nvfp4_quantize ->
 *               out_q [rows_max, N/4] bytes and out_sf = SF(rows_max x N/2)
 *               swizzled; h_debug NULL or fp32 [rows_max, N/2].
 *               NVFP4_EPI_BF16: out_bf16 BF16 [rows_max, N].
 *               NVFP4_EPI_SWIGLU_BF16: h as above, rounded to BF16 into out_bf16
 *               [rows_max, N/2] (out_global_scale does not apply).
 * Two kernels compute this (nvfp4_set_gemm_tiles): 128-row tiles on single CTAs,
 * or, when N % 256 == 0, 256-row tiles on CTA pairs (a 2-CTA cluster sharing one
 * cta_group::2 MMA, each CTA loading half of B), which pairs consecutive 128-row
 * blocks of a group.  With the automatic choice, a grouped GEMM (G > 1, offsets
 * given, no gather) on CTA pairs is split: the single-CTA kernel runs on 8 SMs
 * beside the pair kernel, on a stream of the library's own forked from `stream`
 * and joined back to it through events (so the call stays ordered on `stream`,
 * also under stream capture), and computes the last 128-row block of the
 * thinnest groups with an odd block count, whose half-empty pair tiles the pair
 * kernel then skips.  Every form gives the same results bit for bit.  Every TMA
 * load reads this GPU's memory into the issuing CTA's own shared memory (no
 * cluster multicast).
 * Limits: K a positive multiple of 256, N a positive multiple of 256 (the SwiGLU
 * epilogues) or 128 (BF16), rows_max a
 * positive multiple of 128, all pointers 16-byte aligned.
 * -------------------------------------------------------------------------- */
nvfp4_status nvfp4_grouped_gemm(const uint8_t* a_q, const uint8_t* a_sf, int64_t rows_max,
                                const int32_t* group_offsets, const int32_t* group_counts,
                                int32_t G, int32_t N, int32_t K, const uint8_t* b_q,
                                const uint8_t* b_sf, float alpha, const float* a_global_scale,
                                const float* b_global_scale, const float* out_global_scale,
                                nvfp4_epilogue epilogue, uint8_t* out_q, uint8_t* out_sf,
                                void* out_bf16, float* h_debug, const int32_t* a_gather,
                                int64_t a_gather_rows, const nvfp4_combine_job* side_combine,
                                const nvfp4_stage_job* side_stage, nvfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * nvfp4_mma_peak_probe -- measures the issue ceiling of the block-scaled FP4
 * MMA that the CTA-pair GEMM uses (tcgen05.mma.cta_group::2.kind::mxf4nvf4
 * .block_scale.scale_vec::4X, M=256 N=256 K=64): on every SM pair, `iters`
 * groups of the GEMM's per-K-stage instruction stream (twelve scale-factor
 * copies, four MMAs, one commit) with operands resident in shared memory, no
 * loads and no epilogue.  A measurement aid with no counterpart in the source
 * pages: it gives the GEMMs' roofline the rate of the instruction they issue.
 * The MMA results are discarded.
 *   iters    1 .. 1048576 (each costs ~128 SM cycles x 4 per SM pair)
 *   tflops   out (host): 2*256*256*64 FLOP per MMA over the span from the first
 *            to the last pair's last MMA (globaltimer)
 *   sm_mhz   out (host): the SM clock seen by the issuing threads (clock64 over
 *            globaltimer), mean over the pairs
 * Synchronous: it synchronises `stream` and reads the device error word
 * (NVFP4_ERR_TIMEOUT if a bounded wait gave up).  NVFP4_ERR_INVALID_ARG for a
 * null result pointer or iters out of range.
 * -------------------------------------------------------------------------- */
nvfp4_status nvfp4_mma_peak_probe(int32_t iters, double* tflops, double* sm_mhz, nvfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * nvfp4_set_gemm_tiles -- process-wide choice of nvfp4_grouped_gemm's tile kernel
 * (also used by nvfp4_moe_ffn_forward): NVFP4_GEMM_TILES_AUTO (the default),
 * _SINGLE or _PAIR (_PAIR falls back to single CTAs where N % 256 != 0 or
 * G > 512).  A tuning and testing control with no counterpart in the source
 * pages; results
 * do not depend on it.  Takes effect for calls made after it returns;
 * NVFP4_ERR_INVALID_ARG for another value.
 * -------------------------------------------------------------------------- */
nvfp4_status nvfp4_set_gemm_tiles(int32_t mode);


/* ---------------------------------------------------------------------------
 * nvfp4_moe_ffn_forward -- L1 GEMM with the fused SwiGLU + NVFP4 epilogue, then
 * the L2 GEMM ("NVFP4 MegaMoE Debug Log", "NVFP4 MoE Pipeline"; the fused FP4
 * epilogue planned in "NVFP4-1.1 Approach, Part 2").
 *   a1_q, a1_sf, expert_offsets, expert_counts: as written by moe_route_permute.
 *   w1_q, w1_sf  [E, 2I, H/2] with rows interleaved 8|8 (gate rows, then up rows,
 *                per 16), SF per expert (2I x H).
 *   w2_q, w2_sf  [E, H, I/2], SF per expert (H x I).
 *   a2_q, a2_sf  [rows_max, I/2] and SF(rows_max x I): the re-quantised SwiGLU
 *                output (written for real rows only).
 *   rows_out     BF16 [rows_max, H]: alpha2 * L2 rows (real rows only).
 *   h_debug      NULL or fp32 [rows_max, I] (pre-quantisation h).
 *   x_global_scale, w1_global_scale [E], a2_global_scale, w2_global_scale [E]:
 *                NULL or the two-level encode scales of A1, W1, A2 and W2
 *                (device fp32).  L1 applies alpha1 / (g_x * g_w1[e]) and
 *                re-quantises fp32(h * g_a2); L2 applies alpha2 / (g_a2 * g_w2[e])
 *                (the pages' alpha = igs * global_sf).  g_a2 is an input: the
 *                fused epilogue quantises each tile as it is produced, before the
 *                tensor's amax exists, so the scale is calibrated ahead.
 *   a1_gather, a1_gather_rows  NULL, or L1 gathers its A rows: a1_q is
 *                moe_route_permute's x_q [T, H/2] and a1_gather its perm_token
 *                (a1_gather_rows = T); see nvfp4_grouped_gemm.
 *   prev_combine NULL, or the combine of an EARLIER batch with the same H,
 *                handed to the L1 GEMM as its side_combine (nvfp4_grouped_gemm).
 *                A serving loop then runs route(i), ffn(i) with combine(i-1), and
 *                so on, and one plain moe_combine after the last batch.
 * Limits: H and I positive multiples of 256, rows_max a positive multiple of 128.
 * -------------------------------------------------------------------------- */
nvfp4_status nvfp4_moe_ffn_forward(const uint8_t* a1_q, const uint8_t* a1_sf,
                                   const int32_t* expert_offsets, const int32_t* expert_counts,
                                   int32_t E, int32_t H, int32_t I, int64_t rows_max,
                                   const uint8_t* w1_q, const uint8_t* w1_sf,
                                   const uint8_t* w2_q, const uint8_t* w2_sf, float alpha1,
                                   float alpha2, const float* x_global_scale,
                                   const float* w1_global_scale, const float* a2_global_scale,
                                   const float* w2_global_scale, uint8_t* a2_q, uint8_t* a2_sf,
                                   void* rows_out_bf16, float* h_debug, const int32_t* a1_gather,
                                   int64_t a1_gather_rows, const nvfp4_combine_job* prev_combine,
                                   nvfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_combine -- "scatter with routing weights" ("NVFP4 MegaMoE Debug Log",
 * "NVFP4 MoE Pipeline"): y[t, :] = bf16( sum_{j < top_k} w[t, j] * rows[inv_perm[t, j], :]
 *                                        + shared[t, :] ),
 * accumulated in fp32 in slot order, the shared row last.
 *   rows_bf16   BF16 [*, H]; inv_perm int32 [T, top_k]; topk_w fp32 [T, top_k];
 *   shared_bf16 NULL or BF16 [T, H]: a shared expert's output rows (the pages'
 *               checkpoint notes list a shared expert beside the routed ones).
 *   y_bf16      BF16 [T, H].  H a positive multiple of 8; pointers 16-byte aligned.
 * -------------------------------------------------------------------------- */
nvfp4_status moe_combine(const void* rows_bf16, const int32_t* inv_perm, const float* topk_w,
                         int32_t T, int32_t H, int32_t top_k, const void* shared_bf16,
                         void* y_bf16, nvfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * nvfp4_moe_forward_host -- the whole path for activations and router logits
 * in HOST memory, with the output written back to host memory ("NVFP4 MegaMoE
 * Debug Log", "NVFP4 MoE Pipeline": stage_activation, the two GEMMs and the
 * scatter with routing weights), as one call:
 *   x_host -> buf->x, logits_host -> buf->logits (cudaMemcpyAsync host to
 *   device), moe_route_permute, nvfp4_moe_ffn_forward, moe_combine, then
 *   buf->y -> y_host (device to host), all enqueued on `stream` in that order.
 * The call returns once the work is enqueued; y_host is complete when the
 * stream reaches that point (synchronise the stream or record an event).
 * Host buffers should be pinned (cudaHostAlloc / cudaHostRegister) for the
 * copies to run asynchronously; pageable ones work but the runtime then
 * stages them synchronously.  Overlapping consecutive calls needs two
 * buffer sets on two streams: the copies of one then run beside the other's
 * kernels.
 *   x_host      BF16 [T, H]; logits_host fp32 [T, E]; y_host BF16 [T, H].
 *   w           the expert weights (device): W1 [E, 2I, H/2] + SF, W2 [E, H, I/2] + SF,
 *               as for nvfp4_moe_ffn_forward (one-level scales, alpha 1).
 *   buf         device buffers, as for the three calls it makes: x [T, H] BF16,
 *               logits [T, E], y [T, H], the routing outputs, a1 (permuted
 *               copy) and a2 with their scales, the BF16 L2 rows and the
 *               routing workspace; rows_max = moe_padded_rows_max(T, E, top_k).
 * Limits and errors: those of the calls it makes (checked before anything is
 * enqueued); NVFP4_ERR_INVALID_ARG for a null pointer or T < 1.
 * -------------------------------------------------------------------------- */
typedef struct {
  const uint8_t* w1_q;
  const uint8_t* w1_sf;
  const uint8_t* w2_q;
  const uint8_t* w2_sf;
} nvfp4_moe_weights;

typedef struct {
  void* x_bf16;
  float* logits;
  void* y_bf16;
  int32_t* topk_ids;
  float* topk_w;
  int32_t* expert_counts;
  int32_t* expert_offsets;
  int32_t* perm_token;
  int32_t* inv_perm;
  uint8_t* a1_q;
  uint8_t* a1_sf;
  uint8_t* a2_q;
  uint8_t* a2_sf;
  void* rows_bf16;
  void* workspace;
  size_t workspace_bytes;
  int64_t rows_max;
} nvfp4_moe_buffers;

nvfp4_status nvfp4_moe_forward_host(const void* x_host, const float* logits_host, void* y_host,
                                    int32_t T, int32_t H, int32_t I, int32_t E, int32_t top_k,
                                    const nvfp4_moe_weights* w, const nvfp4_moe_buffers* buf,
                                    nvfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * nvfp4_moe_step_host / nvfp4_moe_finish_host -- a serving loop over batches in
 * host memory, in which each batch's L2 GEMM and combine run in the NEXT step,
 * overlapped with the next batch's work: the L2 GEMM stages the next batch's
 * activation on two spare warps per CTA (nvfp4_grouped_gemm's side_stage), and
 * the next batch's L1 GEMM runs the combine on two spare warps per CTA
 * (side_combine).  One step, enqueued on `stream`:
 *   1. x_host -> buf->x_bf16, logits_host -> buf->logits (host to device);
 *   2. if compute_after is not NULL, wait for it (cudaStreamWaitEvent);
 *   3. without prev: moe_route_permute (with staging) and the L1 GEMM of this
 *      batch into buf.  With prev (the earlier batch, prev_T tokens, whose L2
 *      and combine are pending): moe_route_permute of this batch without
 *      staging, the L2 GEMM of prev staging this batch into buf->a1_q / a1_sf
 *      alongside, then the L1 GEMM of this batch running prev's combine into
 *      prev->y_bf16 alongside;
 *   4. if compute_done is not NULL, record it;
 *   5. if prev is not NULL, prev->y_bf16 -> prev_y_host (device to host).
 * This batch's L2 and combine stay pending in buf: a later step passes buf as
 * its prev, or nvfp4_moe_finish_host runs them (L2, moe_combine, then
 * y -> y_host).  The results equal nvfp4_moe_forward_host's bit for bit.
 * Rotating three buffer sets over three streams, with each step's
 * compute_after the previous step's compute_done, lets the copies of one step
 * run beside the kernels of the next two.  The caller owns the events
 * (cudaEventCreateWithFlags(..., cudaEventDisableTiming) will do) and keeps a
 * set's buffers alive until its y has been copied out.  Arguments as for
 * nvfp4_moe_forward_host; prev, when given, is another buffer set (no buffer
 * shared with buf) for the same H, I, E and top_k.  Everything is checked
 * before anything is enqueued.
 * -------------------------------------------------------------------------- */
typedef struct CUevent_st* nvfp4_event_t;   /* identical to cudaEvent_t */

nvfp4_status nvfp4_moe_step_host(const void* x_host, const float* logits_host, int32_t T, int32_t H,
                                 int32_t I, int32_t E, int32_t top_k, const nvfp4_moe_weights* w,
                                 const nvfp4_moe_buffers* buf, const nvfp4_moe_buffers* prev,
                                 int32_t prev_T, void* prev_y_host, nvfp4_event_t compute_after,
                                 nvfp4_event_t compute_done, nvfp4_stream_t stream);

nvfp4_status nvfp4_moe_finish_host(const nvfp4_moe_weights* w, const nvfp4_moe_buffers* buf, int32_t T,
                                   int32_t H, int32_t I, int32_t E, int32_t top_k, void* y_host,
                                   nvfp4_stream_t stream);

/* Message of the last failing call on this host thread ("" if none). */
const char* nvfp4_last_error(void);

/* Synchronises `stream`, then reads and clears the current device's error word:
 * NVFP4_OK, NVFP4_ERR_TIMEOUT (a bounded wait gave up), NVFP4_ERR_DEVICE (an index
 * check failed) or NVFP4_ERR_CUDA (the stream itself reported an error). */
nvfp4_status nvfp4_device_status(nvfp4_stream_t stream);

/* Self-test of the failure path: launches one warp that waits on *flag (device
 * int32) until it becomes non-zero or `limit_ns` nanoseconds pass, then records a
 * timeout in the error word and returns.  Nothing in the library sets *flag. */
nvfp4_status nvfp4_selftest_bounded_wait(const int32_t* flag, int64_t limit_ns,
                                         nvfp4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4MOE_H */

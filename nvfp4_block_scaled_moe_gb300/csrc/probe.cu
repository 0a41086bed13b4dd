// Measurement of the tensor-core issue ceiling that bounds the NVFP4 GEMMs: the
// block-scaled FP4 MMA of the CTA-pair kernel (tcgen05.mma.cta_group::2
// .kind::mxf4nvf4.block_scale.scale_vec::4X, M=256, N=256, K=64), issued back to
// back with its operands resident in shared memory, on every SM of the GPU.
// Each group of four MMAs is preceded by the twelve scale-factor copies and
// followed by the commit that the GEMM issues per 256-element K stage, so the
// figure is the ceiling of the GEMM's own instruction stream with no loads, no
// hand-off and no epilogue.
//
// Not part of the MoE path: bench.py reports it next to the roofline of the L1
// GEMM so that the measured fraction can be read against the instruction the
// kernel actually issues (the nominal dense FP4/BF16 ratio assumes a faster form).
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "nvfp4moe.h"

namespace nvfp4 {
namespace {

constexpr int kProbeThreads = 128;
constexpr int kProbeMaxCtas = 256;
constexpr uint32_t kProbeSmem = 120 * 1024;     // more than half an SM's shared memory: one CTA per SM
constexpr uint32_t kProbeOffB = 16384, kProbeOffSf = 32768, kProbeOffBar = 40960;

// per CTA: globaltimer at the first and after the last MMA, clock64 likewise
__device__ unsigned long long g_probe_stamps[4 * kProbeMaxCtas];

__global__ void __launch_bounds__(kProbeThreads, 1) mma_probe_kernel(int32_t iters, unsigned* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  // the swizzled operand tiles need a 1 KiB-aligned base; every CTA sees the
  // same base, so a misaligned one stops all of them before any pair traffic
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) raise_error(err, kErrBounds);
    return;
  }
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kProbeOffBar);     // [0] final commit, [1] per-stage commits
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kProbeOffBar + 64);
  const int warp = threadIdx.x >> 5;
  const uint32_t rank = cluster_ctarank();

  // operands: any byte is a finite pair of E2M1 values; scale codes 0x38 = 1.0
  uint32_t h = 0x9E3779B9u * (blockIdx.x + 1);
  for (int i = threadIdx.x; i < static_cast<int>(kProbeOffSf / 4); i += blockDim.x) {
    uint32_t v = (static_cast<uint32_t>(i) + 1u) * 2654435761u ^ h;
    v ^= v >> 13;
    v *= 0x5bd1e995u;
    v ^= v >> 15;
    reinterpret_cast<uint32_t*>(smem)[i] = v;
  }
  for (int i = threadIdx.x; i < 8192 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(smem + kProbeOffSf)[i] = 0x38383838u;
  fence_async_smem();                        // the generic-proxy writes above are read by the MMA
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    unsigned long long t0 = 0, c0 = 0;
    if (rank == 0 && elect_one()) {
      constexpr uint32_t idesc = idesc_nvf4(256, 256);
      const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(smem));
      const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(smem + kProbeOffB));
      const uint32_t sf_s = smem_u32(smem + kProbeOffSf);
      t0 = globaltimer_ns();
      c0 = clock64();
      uint32_t stage = 0;
      for (int32_t it = 0; it < iters; ++it) {
        const uint32_t sfa_t = tmem + 256 + stage * 48, sfb_t = sfa_t + 16;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          tc_copy_sf_pair(sfa_t + 4 * j, sdesc_sf(sf_s + 512 * j));
#pragma unroll
          for (int b = 0; b < 2; ++b) tc_copy_sf_pair(sfb_t + 8 * j + 4 * b, sdesc_sf(sf_s + 2048 + 2048 * b + 512 * j));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          tc_mma_nvf4_pair(tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sfa_t + 4 * j, sfb_t + 8 * j,
                           (it | j) != 0 ? 1u : 0u);
        tc_commit_pair_mc(&bar[1], 0x3);
        if (++stage == 5) stage = 0;
      }
      tc_commit_pair_mc(&bar[0], 0x3);
    }
    __syncwarp();
    int no_abort = 0;
    const bool ok = mbar_wait(&bar[0], 0, &no_abort, err, 2000000000ull);
    if (rank == 0 && ok && (threadIdx.x & 31) == 0 && blockIdx.x < kProbeMaxCtas) {   // the issuing lane
      unsigned long long* st = g_probe_stamps + 4 * blockIdx.x;
      st[0] = t0;
      st[1] = globaltimer_ns();
      st[2] = c0;
      st[3] = clock64();
    }
    __syncwarp();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();          // neither CTA frees TMEM while the pair's MMAs may still run
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status nvfp4_mma_peak_probe(int32_t iters, double* tflops, double* sm_mhz, nvfp4_stream_t stream) {
  if (tflops == nullptr || sm_mhz == nullptr)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_mma_peak_probe: null result pointer");
  if (iters < 1 || iters > (1 << 20))
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_mma_peak_probe: iters=%d outside [1, 1048576]", iters);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(mma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kProbeSmem));
  if (e != cudaSuccess) return fail_cuda(e, "nvfp4_mma_peak_probe: setup");
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kProbeThreads, 1, 1);
  cfg.gridDim = dim3(static_cast<unsigned>(std::min(sms, kProbeMaxCtas) & ~1), 1, 1);
  cfg.dynamicSmemBytes = kProbeSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, mma_probe_kernel, &cfg);
  if (e != cudaSuccess) return fail_cuda(e, "nvfp4_mma_peak_probe: occupancy");
  clusters = std::min(clusters, kProbeMaxCtas / 2);
  if (clusters <= 0) return fail(NVFP4_ERR_CUDA, "nvfp4_mma_peak_probe: no resident cluster");
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
  void* stamps = nullptr;
  e = cudaGetSymbolAddress(&stamps, g_probe_stamps);
  if (e == cudaSuccess) e = cudaMemsetAsync(stamps, 0, sizeof(unsigned long long) * 4 * kProbeMaxCtas, s);
  if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, mma_probe_kernel, iters, device_error_word());
  unsigned long long host[4 * kProbeMaxCtas];
  if (e == cudaSuccess) e = cudaMemcpyAsync(host, stamps, sizeof(host), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e, "nvfp4_mma_peak_probe: run");
  const nvfp4_status st = nvfp4_device_status(stream);
  if (st != NVFP4_OK) return st;
  unsigned long long t_lo = ~0ull, t_hi = 0;
  double mhz = 0.0;
  int n = 0;
  for (int c = 0; c < clusters; ++c) {
    const unsigned long long* p = host + 4 * (2 * c);
    if (p[1] == 0 || p[1] <= p[0]) continue;
    t_lo = std::min(t_lo, p[0]);
    t_hi = std::max(t_hi, p[1]);
    mhz += static_cast<double>(p[3] - p[2]) / static_cast<double>(p[1] - p[0]) * 1e3;
    ++n;
  }
  if (n != clusters) return fail(NVFP4_ERR_CUDA, "nvfp4_mma_peak_probe: %d of %d clusters reported", n, clusters);
  const double flop = 2.0 * 256 * 256 * 64 * 4.0 * iters * clusters;
  *tflops = flop / static_cast<double>(t_hi - t_lo) / 1e3;
  *sm_mhz = mhz / n;
  return NVFP4_OK;
}

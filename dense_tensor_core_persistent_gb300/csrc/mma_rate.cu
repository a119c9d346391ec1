// mma_rate.cu -- gemm_measure_mma_rate: the throughput of the two tensor-core MMA kinds
// the GEMMs issue, in FLOP per SM clock, measured on the current GPU.
//
// One CTA pair per two SMs; the leader thread issues back-to-back M = 256, N = 256 MMAs
// (cta_group::2) into one TMEM accumulator from shared-memory operands, with nothing
// else to wait for, and times them with the SM clock. This is the instruction ceiling a
// GEMM kernel of that shape can approach: kind::f16 (BF16, K = 16) and
// kind::mxf4nvf4.block_scale.scale_vec::4X (E2M1 with UE4M3 scales, K = 64).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "gemm.h"
#include "host_common.h"

namespace dtcp {
namespace {

constexpr int kRateThreads = 128;
constexpr int kRateOperandBytes = 64 * 1024;               // A at 0, B at 32 KB
// more shared memory than two CTAs can share on one SM: one CTA (and one TMEM owner) per SM
constexpr int kRateSmem = 128 * 1024;
constexpr int kRateMaxClusters = 256;

// Cycles each cluster's leader thread spent on its MMAs (one entry per cluster).
static __device__ unsigned long long g_rate_cycles[kRateMaxClusters];

template <int KIND>
__global__ void __launch_bounds__(kRateThreads, 1) mma_rate_kernel(int iters, unsigned* status,
                                                                    unsigned long long wait_limit_ns) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t bar_done = base + kRateOperandBytes;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kRateOperandBytes + 64);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kRateOperandBytes + 128);

  for (int i = threadIdx.x; i < kRateOperandBytes / 16; i += blockDim.x) st_shared_v4(base + 16 * i, 0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    mbar_init(bar_done, 1);
    *abort_flag = 0u;
    fence_mbarrier_init_cluster();
  }
  fence_proxy_async_smem();  // zeroed operands are read by the tensor cores (async proxy)
  if (warp == 1) {
    tmem_alloc<2>(smem_u32(tmem_slot), 512);
    tmem_relinquish<2>();
  }
  tc_fence_before_sync();
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0 && rank == 0) {
    const uint64_t a = umma_desc_sw128(base), b = umma_desc_sw128(base + kRateOperandBytes / 2);
    const unsigned long long t0 = clock64();
    for (int i = 0; i < iters; i += 4) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if constexpr (KIND == 0)
          mma_f16<2>(tmem, umma_desc_advance(a, 32 * j), umma_desc_advance(b, 32 * j), idesc_bf16(256, 256),
                     (i | j) != 0 ? 1u : 0u);
        else
          mma_nvf4<2>(tmem, umma_desc_advance(a, 32 * j), umma_desc_advance(b, 32 * j), idesc_nvf4(256, 256),
                      tmem + 256 + 4 * j, tmem + 272 + 8 * j, (i | j) != 0 ? 1u : 0u);
      }
    }
    // the clock stops when the last MMA has completed
    mma_commit_pair_multicast(bar_done, 0x1);
    const WaitCtx w{abort_flag, status, wait_limit_ns};
    wait_phase_slow(bar_done, 0, w, status_code(kRoleMma, 0xFFFD), false);
    g_rate_cycles[blockIdx.x / 2] = clock64() - t0;
  }
  __syncwarp();
  tc_fence_before_sync();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc<2>(tmem, 512);
  }
}

template <int KIND>
int run_rate(int device, const DeviceInfo& info, int iters, double* flop_per_clock) {
  const auto kernel = mma_rate_kernel<KIND>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRateSmem) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  unsigned* status = device_status_word(device);
  if (status == nullptr) return GEMM_ERR_NO_DEVICE;
  int clusters = info.num_sms / 2;
  if (clusters > kRateMaxClusters) clusters = kRateMaxClusters;
  if (clusters < 1) return GEMM_ERR_NO_DEVICE;
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
  cfg.blockDim = dim3(kRateThreads, 1, 1);
  cfg.dynamicSmemBytes = kRateSmem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const unsigned long long limit = 2000000000ull;
  int st = GEMM_OK;
  for (int rep = 0; rep < 2 && st == GEMM_OK; ++rep) {  // the first launch warms up clocks and caches
    if (cudaLaunchKernelEx(&cfg, kernel, iters, status, limit) != cudaSuccess) st = GEMM_ERR_LAUNCH;
    else count_launch();
  }
  if (cudaStreamSynchronize(s) != cudaSuccess) st = GEMM_ERR_LAUNCH;
  unsigned long long cyc[kRateMaxClusters] = {0};
  if (st == GEMM_OK && cudaMemcpyFromSymbol(cyc, g_rate_cycles, sizeof(unsigned long long) * clusters) != cudaSuccess)
    st = GEMM_ERR_LAUNCH;
  cudaStreamDestroy(s);
  if (st != GEMM_OK) {
    cudaGetLastError();
    return st;
  }
  unsigned word = 0;
  if (cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return GEMM_ERR_LAUNCH;
  if ((word & 0xFFu) == GEMM_ERR_TIMEOUT) return GEMM_ERR_TIMEOUT;
  double mean = 0.0;
  for (int c = 0; c < clusters; ++c) mean += static_cast<double>(cyc[c]);
  mean /= clusters;
  if (mean <= 0.0) return GEMM_ERR_LAUNCH;
  // FLOP of one M = 256, N = 256 MMA per SM of the pair: 2 * 128 * 256 * K
  const double k = KIND == 0 ? 16.0 : 64.0;
  *flop_per_clock = static_cast<double>(iters) * 2.0 * 128.0 * 256.0 * k / mean;
  return GEMM_OK;
}

}  // namespace
}  // namespace dtcp

using namespace dtcp;

extern "C" int gemm_measure_mma_rate(int kind, double* flop_per_clock_per_sm) {
  if (flop_per_clock_per_sm == nullptr || (kind != GEMM_MMA_BF16 && kind != GEMM_MMA_NVFP4)) return GEMM_ERR_INVALID_ARG;
  int device = 0, err = 0;
  const DeviceInfo* info = current_device_info(&device, &err);
  if (info == nullptr) return err;
  const int iters = 8192;  // about a million SM clocks per launch
  return kind == GEMM_MMA_BF16 ? run_rate<0>(device, *info, iters, flop_per_clock_per_sm)
                               : run_rate<1>(device, *info, iters, flop_per_clock_per_sm);
}

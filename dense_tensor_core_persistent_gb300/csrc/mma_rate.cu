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
constexpr int kRateMaxCtas = 256;

// Cycles each issuing thread spent on its MMAs (one entry per issuing CTA).
static __device__ unsigned long long g_rate_cycles[kRateMaxCtas];

// The instruction forms measured. CG: CTAs per MMA (2 = a pair, M = 256; 1 = M = 128).
// ACCS: accumulators the MMAs alternate between (columns 0 and N). K: per instruction.
// FORM: 0 kind::f16 (BF16), 1 kind::mxf4nvf4 scale_vec::4X (UE4M3 per 16),
// 2 kind::mxf4 scale_vec::2X (UE8M0 per 32).
struct RateForm {
  int cg, n, accs, k, form;
};

__host__ __device__ constexpr RateForm rate_form(int kind) {
  switch (kind) {
    case GEMM_MMA_BF16: return RateForm{2, 256, 1, 16, 0};
    case GEMM_MMA_NVFP4: return RateForm{2, 256, 1, 64, 1};
    case GEMM_MMA_NVFP4_1CTA_N128: return RateForm{1, 128, 1, 64, 1};
    case GEMM_MMA_NVFP4_1CTA_N192: return RateForm{1, 192, 1, 64, 1};
    case GEMM_MMA_NVFP4_1CTA_N256: return RateForm{1, 256, 1, 64, 1};
    case GEMM_MMA_NVFP4_PAIR_N128: return RateForm{2, 128, 1, 64, 1};
    case GEMM_MMA_NVFP4_PAIR_N128_2ACC: return RateForm{2, 128, 2, 64, 1};
    case GEMM_MMA_MXF4_PAIR_N256: return RateForm{2, 256, 1, 64, 2};
    default: return RateForm{0, 0, 0, 0, -1};
  }
}

// Block-scaled instruction descriptor with UE8M0 scales (bit 23 = 1), E2M1 operands:
// kind::mxf4 with one scale per 32 K-elements.
__host__ __device__ constexpr uint32_t idesc_mxf4(int m, int n) { return idesc_nvf4(m, n) | (1u << 23); }

template <int CG>
__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  if constexpr (CG == 1)
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// One issuing thread per MMA group (the pair's leader, or every CTA for CG = 1) issues
// `iters` MMAs of the form back to back on zeroed operands. The scale factors sit in
// columns 384.. (at most 4 MMAs x (4 + 8) columns); accumulators at 0 and N.
template <int KIND>
__global__ void __launch_bounds__(kRateThreads, 1) mma_rate_kernel(int iters, unsigned* status,
                                                                    unsigned long long wait_limit_ns) {
  constexpr RateForm F = rate_form(KIND);
  constexpr int CG = F.cg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
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
    tmem_alloc<CG>(smem_u32(tmem_slot), 512);
    tmem_relinquish<CG>();
  }
  tc_fence_before_sync();
  if constexpr (CG == 2) cluster_sync_all();
  else __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0 && rank == 0) {
    const uint64_t a = umma_desc_sw128(base), b = umma_desc_sw128(base + kRateOperandBytes / 2);
    const uint32_t sf = tmem + 384;
    const unsigned long long t0 = clock64();
    for (int i = 0; i < iters; i += 4) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t d = tmem + (F.accs == 2 ? static_cast<uint32_t>(j & 1) * F.n : 0u);
        const uint32_t acc = (i != 0 || j >= F.accs) ? 1u : 0u;
        if constexpr (F.form == 0)
          mma_f16<CG>(d, umma_desc_advance(a, 32 * j), umma_desc_advance(b, 32 * j), idesc_bf16(128 * CG, F.n), acc);
        else if constexpr (F.form == 1)
          mma_nvf4<CG>(d, umma_desc_advance(a, 32 * j), umma_desc_advance(b, 32 * j), idesc_nvf4(128 * CG, F.n),
                       sf + 4 * j, sf + 16 + 8 * j, acc);
        else
          mma_mxf4<CG>(d, umma_desc_advance(a, 32 * j), umma_desc_advance(b, 32 * j), idesc_mxf4(128 * CG, F.n),
                       sf + 4 * j, sf + 16 + 8 * j, acc);
      }
    }
    // the clock stops when the last MMA has completed
    if constexpr (CG == 2) mma_commit_pair_multicast(bar_done, 0x1);
    else mma_commit_local(bar_done);
    const WaitCtx w{abort_flag, status, wait_limit_ns};
    wait_phase_slow(bar_done, 0, w, status_code(kRoleMma, 0xFFFD), false);
    g_rate_cycles[blockIdx.x / CG] = clock64() - t0;
  }
  __syncwarp();
  tc_fence_before_sync();
  if constexpr (CG == 2) cluster_sync_all();
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc<CG>(tmem, 512);
  }
}

template <int KIND>
int run_rate(int device, const DeviceInfo& info, int iters, double* flop_per_clock) {
  constexpr RateForm F = rate_form(KIND);
  const auto kernel = mma_rate_kernel<KIND>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRateSmem) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  unsigned* status = device_status_word(device);
  if (status == nullptr) return GEMM_ERR_NO_DEVICE;
  int groups = info.num_sms / F.cg;  // one issuing CTA per SM pair (CG = 2) or per SM
  if (groups > kRateMaxCtas) groups = kRateMaxCtas;
  if (groups < 1) return GEMM_ERR_NO_DEVICE;
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(static_cast<unsigned>(F.cg * groups), 1, 1);
  cfg.blockDim = dim3(kRateThreads, 1, 1);
  cfg.dynamicSmemBytes = kRateSmem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = F.cg;
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
  unsigned long long cyc[kRateMaxCtas] = {0};
  if (st == GEMM_OK && cudaMemcpyFromSymbol(cyc, g_rate_cycles, sizeof(unsigned long long) * groups) != cudaSuccess)
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
  for (int c = 0; c < groups; ++c) mean += static_cast<double>(cyc[c]);
  mean /= groups;
  if (mean <= 0.0) return GEMM_ERR_LAUNCH;
  // FLOP of one MMA per SM: 2 * 128 * N * K (a pair's M = 256 spans two SMs)
  *flop_per_clock = static_cast<double>(iters) * 2.0 * 128.0 * F.n * F.k / mean;
  return GEMM_OK;
}

}  // namespace
}  // namespace dtcp

using namespace dtcp;

extern "C" int gemm_measure_mma_rate(int kind, double* flop_per_clock_per_sm) {
  if (flop_per_clock_per_sm == nullptr || rate_form(kind).form < 0) return GEMM_ERR_INVALID_ARG;
  int device = 0, err = 0;
  const DeviceInfo* info = current_device_info(&device, &err);
  if (info == nullptr) return err;
  const int iters = 8192;  // about a million SM clocks per launch
  double* r = flop_per_clock_per_sm;
  switch (kind) {
    case GEMM_MMA_BF16: return run_rate<GEMM_MMA_BF16>(device, *info, iters, r);
    case GEMM_MMA_NVFP4: return run_rate<GEMM_MMA_NVFP4>(device, *info, iters, r);
    case GEMM_MMA_NVFP4_1CTA_N128: return run_rate<GEMM_MMA_NVFP4_1CTA_N128>(device, *info, iters, r);
    case GEMM_MMA_NVFP4_1CTA_N192: return run_rate<GEMM_MMA_NVFP4_1CTA_N192>(device, *info, iters, r);
    case GEMM_MMA_NVFP4_1CTA_N256: return run_rate<GEMM_MMA_NVFP4_1CTA_N256>(device, *info, iters, r);
    case GEMM_MMA_NVFP4_PAIR_N128: return run_rate<GEMM_MMA_NVFP4_PAIR_N128>(device, *info, iters, r);
    case GEMM_MMA_NVFP4_PAIR_N128_2ACC: return run_rate<GEMM_MMA_NVFP4_PAIR_N128_2ACC>(device, *info, iters, r);
    case GEMM_MMA_MXF4_PAIR_N256: return run_rate<GEMM_MMA_MXF4_PAIR_N256>(device, *info, iters, r);
    default: return GEMM_ERR_INVALID_ARG;
  }
}

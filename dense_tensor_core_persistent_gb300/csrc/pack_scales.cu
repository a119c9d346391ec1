// pack_scales.cu -- rearrange NVFP4 scale factors from row-major [rows][K/16] into the
// blocked layout the block-scaled tensor-core MMA reads through tcgen05.cp.
//
// Blocked layout (for `rows` rows and K columns, K % 64 == 0): rows are padded to a
// multiple of 128; block (rb, j) covers rows 128 rb .. 128 rb + 127 and K elements
// 64 j .. 64 j + 63 (four 16-element scale groups) and is 512 contiguous bytes at offset
// (rb * K/64 + j) * 512. Inside a block, the 16-byte line l (l < 32) holds the four
// scales of rows l, l+32, l+64, l+96 in that order, each as 4 bytes for the 16-element
// groups 0..3 of the 64-K step. A `.32x128b.warpx4` copy of one block puts line l into
// TMEM lane l of every 32-lane quadrant, and the MMA rows of quadrant q read column q.
// Padding rows are zero.
//
// ("NVFP4 GEMM on Blackwell", Kernel 1, "Tensor Cores and Tensor Memory": scales live in
// TMEM for the MMA and are moved there with tcgen05.cp .32x128b.warpx4, which copies 32
// lanes x 128 bits and replicates them into all four warps' lane quadrants.)
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "host_common.h"
#include "ptx.cuh"
#include "schedule.h"

namespace dtcp {

constexpr int kPackRows = 128;    // one row block per CTA
constexpr int kPackSteps = 16;    // 64-K steps per CTA (64 scale bytes per row)
constexpr int kPackThreads = 256;

// CTA (x, y): K steps 16 x .. 16 x + 15 of row block y of the first matrix, or of row
// block y - rb0 of the second one (two matrices in one launch). CTAs with y past both
// matrices' row blocks copy `copy_bytes` (a multiple of 16) from copy_src to copy_dst
// instead: the few rows of A that the GEMM reads from a padded buffer.
// VEC16: the scale rows are 16-byte aligned (K % 256 == 0), so each thread reads four
// 64-K steps of a row with one 16-byte load.
template <bool VEC16>
__global__ void __launch_bounds__(kPackThreads) pack_scales_kernel(const uint8_t* __restrict__ sf0,
                                                                   uint8_t* __restrict__ out0, int rows0,
                                                                   const uint8_t* __restrict__ sf1,
                                                                   uint8_t* __restrict__ out1, int rows1,
                                                                   int row_bytes, int ksteps,
                                                                   const uint8_t* __restrict__ copy_src,
                                                                   uint8_t* __restrict__ copy_dst,
                                                                   long long copy_bytes) {
  __shared__ uint32_t tile[kPackRows][kPackSteps + 1];  // +1 word: conflict-free column reads
  const int rb0 = (rows0 + kPackRows - 1) / kPackRows;
  const int rb1 = (rows1 + kPackRows - 1) / kPackRows;
  pdl_launch_dependents();
  pdl_wait();  // the scales (and A) may come from the previous kernel on the stream
  if (static_cast<int>(blockIdx.y) >= rb0 + rb1) {
    const uint4* __restrict__ src = reinterpret_cast<const uint4*>(copy_src);
    uint4* __restrict__ dst = reinterpret_cast<uint4*>(copy_dst);
    const long long n = copy_bytes / 16;
    for (long long i = static_cast<long long>(blockIdx.x) * kPackThreads + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kPackThreads)
      dst[i] = src[i];
    return;
  }
  const bool second = static_cast<int>(blockIdx.y) >= rb0;
  const uint8_t* __restrict__ sf = second ? sf1 : sf0;
  uint8_t* __restrict__ out = second ? out1 : out0;
  const int rows = second ? rows1 : rows0;
  const int rb = second ? static_cast<int>(blockIdx.y) - rb0 : static_cast<int>(blockIdx.y);
  const int j0 = blockIdx.x * kPackSteps;
  const int nj = min(kPackSteps, ksteps - j0);
  if constexpr (VEC16) {
    // 16 bytes (four 64-K steps) of a row per thread and load; nj is a multiple of 4
    for (int i = threadIdx.x; i < kPackRows * (kPackSteps / 4); i += kPackThreads) {
      const int r = i / (kPackSteps / 4), c = i % (kPackSteps / 4);
      const int row = rb * kPackRows + r;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (row < rows && 4 * c < nj)
        v = *reinterpret_cast<const uint4*>(sf + static_cast<size_t>(row) * row_bytes + (j0 + 4 * c) * 4);
      tile[r][4 * c] = v.x;
      tile[r][4 * c + 1] = v.y;
      tile[r][4 * c + 2] = v.z;
      tile[r][4 * c + 3] = v.w;
    }
  } else {
    for (int i = threadIdx.x; i < kPackRows * kPackSteps; i += kPackThreads) {
      const int r = i / kPackSteps, w = i % kPackSteps;
      const int row = rb * kPackRows + r;
      uint32_t v = 0;
      if (row < rows && w < nj)
        v = *reinterpret_cast<const uint32_t*>(sf + static_cast<size_t>(row) * row_bytes + (j0 + w) * 4);
      tile[r][w] = v;
    }
  }
  __syncthreads();
  // nj consecutive 512-byte blocks are contiguous in the output: one 16-byte line per thread
  uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(rb) * ksteps + j0) * 512);
  for (int i = threadIdx.x; i < nj * 32; i += kPackThreads) {
    const int j = i >> 5, l = i & 31;
    dst[i] = make_uint4(tile[l][j], tile[l + 32][j], tile[l + 64][j], tile[l + 96][j]);
  }
}

// The scales of both matrices (either may have 0 rows) and, with copy_bytes > 0, the copy
// of A's rows, in one launch.
static int launch_pack(const void* SF0, void* out0, int rows0, const void* SF1, void* out1, int rows1, int K,
                       const void* copy_src, void* copy_dst, long long copy_bytes, cudaStream_t stream, int pdl) {
  const int ksteps = K / 64;
  const int blocks_y = ceil_div(rows0, kPackRows) + ceil_div(rows1, kPackRows) + (copy_bytes > 0 ? 1 : 0);
  int blocks_x = ceil_div(ksteps, kPackSteps);
  if (copy_bytes > 0) {
    // the copy row of CTAs: enough threads for one 16-byte piece each, within the row's width
    const long long want = (copy_bytes / 16 + kPackThreads - 1) / kPackThreads;
    blocks_x = std::max(blocks_x, static_cast<int>(std::min<long long>(want, 64)));
  }
  if (blocks_x < 1 || blocks_y < 1) return GEMM_OK;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(static_cast<unsigned>(blocks_x), static_cast<unsigned>(blocks_y), 1);
  cfg.blockDim = dim3(kPackThreads, 1, 1);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int row_bytes = K / 16;
  const auto kernel = row_bytes % 16 == 0 ? pack_scales_kernel<true> : pack_scales_kernel<false>;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<const uint8_t*>(SF0), static_cast<uint8_t*>(out0),
                                           rows0, static_cast<const uint8_t*>(SF1), static_cast<uint8_t*>(out1), rows1,
                                           row_bytes, ksteps, static_cast<const uint8_t*>(copy_src),
                                           static_cast<uint8_t*>(copy_dst), copy_bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  count_launch();
  return GEMM_OK;
}

int run_pack_scales2(const void* SF0, void* out0, int rows0, const void* SF1, void* out1, int rows1, int K,
                     cudaStream_t stream, int pdl) {
  return launch_pack(SF0, out0, rows0, SF1, out1, rows1, K, nullptr, nullptr, 0, stream, pdl);
}

int run_pack_scales2_copy(const void* SF0, void* out0, int rows0, const void* SF1, void* out1, int rows1, int K,
                          const void* copy_src, void* copy_dst, long long copy_bytes, cudaStream_t stream, int pdl) {
  return launch_pack(SF0, out0, rows0, SF1, out1, rows1, K, copy_src, copy_dst, copy_bytes, stream, pdl);
}

int run_copy_rows(void* dst, const void* A, int M, int K, cudaStream_t stream, int pdl) {
  return launch_pack(nullptr, nullptr, 0, nullptr, nullptr, 0, K, A, dst,
                     static_cast<long long>(M) * (static_cast<long long>(K) / 2), stream, pdl);
}

int run_pack_scales(const void* SF, void* SF_blocked, int rows, int K, cudaStream_t stream, int pdl) {
  return run_pack_scales2(SF, SF_blocked, rows, nullptr, nullptr, 0, K, stream, pdl);
}

}  // namespace dtcp

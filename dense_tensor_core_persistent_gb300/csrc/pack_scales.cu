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

#include <cstdint>

#include "host_common.h"
#include "ptx.cuh"
#include "schedule.h"

namespace dtcp {

constexpr int kPackRows = 128;    // one row block per CTA
constexpr int kPackSteps = 16;    // 64-K steps per CTA (64 scale bytes per row)
constexpr int kPackThreads = 256;

// CTA (x, y): K steps 16 x .. 16 x + 15 of row block y of the first matrix, or of row
// block y - rb0 of the second one (two matrices in one launch).
__global__ void __launch_bounds__(kPackThreads) pack_scales_kernel(const uint8_t* __restrict__ sf0,
                                                                   uint8_t* __restrict__ out0, int rows0,
                                                                   const uint8_t* __restrict__ sf1,
                                                                   uint8_t* __restrict__ out1, int rows1,
                                                                   int row_bytes, int ksteps) {
  __shared__ uint32_t tile[kPackRows][kPackSteps + 1];  // +1 word: conflict-free column reads
  const int rb0 = (rows0 + kPackRows - 1) / kPackRows;
  const bool second = static_cast<int>(blockIdx.y) >= rb0;
  const uint8_t* __restrict__ sf = second ? sf1 : sf0;
  uint8_t* __restrict__ out = second ? out1 : out0;
  const int rows = second ? rows1 : rows0;
  const int rb = second ? static_cast<int>(blockIdx.y) - rb0 : static_cast<int>(blockIdx.y);
  const int j0 = blockIdx.x * kPackSteps;
  const int nj = min(kPackSteps, ksteps - j0);
  pdl_launch_dependents();
  pdl_wait();  // the scales may come from the previous kernel on the stream
  for (int i = threadIdx.x; i < kPackRows * kPackSteps; i += kPackThreads) {
    const int r = i / kPackSteps, w = i % kPackSteps;
    const int row = rb * kPackRows + r;
    uint32_t v = 0;
    if (row < rows && w < nj)
      v = *reinterpret_cast<const uint32_t*>(sf + static_cast<size_t>(row) * row_bytes + (j0 + w) * 4);
    tile[r][w] = v;
  }
  __syncthreads();
  // nj consecutive 512-byte blocks are contiguous in the output: one 16-byte line per thread
  uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(rb) * ksteps + j0) * 512);
  for (int i = threadIdx.x; i < nj * 32; i += kPackThreads) {
    const int j = i >> 5, l = i & 31;
    dst[i] = make_uint4(tile[l][j], tile[l + 32][j], tile[l + 64][j], tile[l + 96][j]);
  }
}

int run_pack_scales2(const void* SF0, void* out0, int rows0, const void* SF1, void* out1, int rows1, int K,
                     cudaStream_t stream, int pdl) {
  const int ksteps = K / 64;
  const int blocks_y = ceil_div(rows0, kPackRows) + ceil_div(rows1, kPackRows);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(ksteps, kPackSteps)), static_cast<unsigned>(blocks_y), 1);
  cfg.blockDim = dim3(kPackThreads, 1, 1);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, pack_scales_kernel, static_cast<const uint8_t*>(SF0), static_cast<uint8_t*>(out0), rows0,
                         static_cast<const uint8_t*>(SF1), static_cast<uint8_t*>(out1), rows1, K / 16, ksteps);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  count_launch();
  return GEMM_OK;
}

int run_pack_scales(const void* SF, void* SF_blocked, int rows, int K, cudaStream_t stream, int pdl) {
  return run_pack_scales2(SF, SF_blocked, rows, nullptr, nullptr, 0, K, stream, pdl);
}

}  // namespace dtcp

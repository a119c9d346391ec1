// host_common.h -- host-side helpers shared by the launchers and the C ABI (api.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm.h"

namespace dtcp {

// Per-device facts, queried once.
struct DeviceInfo {
  int cc_major = 0;
  int cc_minor = 0;
  int num_sms = 0;
  long long l2_bytes = 0;
  int max_smem_optin = 0;
};

// Current device's facts; nullptr (and *err set) if the runtime call fails.
const DeviceInfo* current_device_info(int* device, int* err);

// cuTensorMapEncodeTiled, reached through the runtime's driver entry point (no -lcuda).
int encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner_elems,
                   uint64_t outer_rows, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                   CUtensorMapSwizzle swizzle);
// 3-D map: dims[0] innermost (elements), strides of dims 1 and 2 in bytes.
int encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, const uint64_t dims[3],
                   const uint64_t strides_bytes[2], const uint32_t box[3],
                   CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE);

// Device address of the process-wide status word on the current device.
unsigned* device_status_word(int device);

void count_launch();

// Resolved per-call options.
// Fused epilogue of the *_fused calls: C = act(alpha * acc + beta * C_old + bias[col]).
struct EpilogueOptions {
  float alpha = 1.0f;
  float beta = 0.0f;
  const void* bias = nullptr;  // N BF16 values, or null
  int act = 0;                 // 0 none, 1 ReLU, 2 GELU (tanh form)
  bool fused() const { return alpha != 1.0f || beta != 0.0f || bias != nullptr || act != 0; }
};

struct RunOptions {
  int kernel = GEMM_KERNEL_DEFAULT;
  int persistent = 1;
  int group_m = 0;
  int max_clusters = 0;
  int tail_split = 1;
  int pdl = 1;  // programmatic stream serialization on the launch
  int swap_ab = 1;  // allow C^T = B A^T for BF16 GEMMs with few rows
  int split_k = 1;  // allow K splits for the swapped BF16 GEMMs
  int clc = 0;      // cluster launch control: 0 = by clc_rule, 1 = on, 2 = off
  int pad_a = 1;    // NVFP4 with 1 <= M < kNvfp4PadRows: read A from a padded copy
  unsigned long long* clock_probe = nullptr;  // gemm_options_t.clock_probe (GEMM kernels only)
  int clock_probe_ctas = 0;
  uint64_t wait_limit_ns = 2000000000ull;
  uint32_t debug_flags = 0;
  EpilogueOptions epi;
};

// The library's stream-ordered memory pool for temporary workspaces (one per device).
cudaMemPool_t workspace_pool(int device);

int run_gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K, cudaStream_t stream,
                  const RunOptions& opt);
// The 512 x 256 pair tile (two M-waves per CTA); plain epilogue, static schedule.
int run_gemm_bf16_wide(const void* A, const void* B, void* C, int M, int N, int K, cudaStream_t stream,
                       const RunOptions& opt);
// Whether run_gemm_bf16 computes C^T = B A^T for this problem, and the tile N it uses.
bool bf16_swap_ab(int M, int N, const RunOptions& opt);
// Whether the default kernel runs this (unswapped) GEMM on the 512 x 256 pair tile, with
// `wave` co-resident clusters.
bool bf16_use_wide(int M, int N, int K, const RunOptions& opt, int wave);
int bf16_tile_n(int M, int N, const RunOptions& opt);
// a_rows: rows of the buffer A points to (>= M): the A tensor map spans them, rows past M
// reach only C rows that are never stored.
int run_gemm_nvfp4_blocked(const void* A, const void* SFA_blocked, const void* B, const void* SFB_blocked, void* C,
                           int M, int N, int K, cudaStream_t stream, const RunOptions& opt, int a_rows = 0);

// NVFP4 GEMMs with fewer rows than this read A from a copy padded to this many rows (see
// gemm_options_t.no_pad_a): measured on GB300, all-CTA reads of an A that spans less than
// 32 rows of 4 KB contend for a few L2 slices.
constexpr int kNvfp4PadRows = 32;
inline int nvfp4_a_rows(int M, const RunOptions& opt) { return (opt.pad_a && M >= 1 && M < kNvfp4PadRows) ? kNvfp4PadRows : M; }
int run_pack_scales(const void* SF, void* SF_blocked, int rows, int K, cudaStream_t stream, int pdl = 1);
// Both matrices of a GEMM in one launch (rows0 + rows1 row blocks).
int run_pack_scales2(const void* SF0, void* out0, int rows0, const void* SF1, void* out1, int rows1, int K,
                     cudaStream_t stream, int pdl = 1);

// The same, plus a copy of copy_bytes (a multiple of 16) from copy_src to copy_dst by extra
// CTAs of the launch (the few rows of A that the GEMM reads from a padded buffer).
int run_pack_scales2_copy(const void* SF0, void* out0, int rows0, const void* SF1, void* out1, int rows1, int K,
                          const void* copy_src, void* copy_dst, long long copy_bytes, cudaStream_t stream, int pdl = 1);
// Copy of M rows of packed E2M1 codes (K / 2 bytes each, K % 256 == 0) by a kernel launched
// with programmatic stream serialization (the GEMM after it starts its set-up early).
int run_copy_rows(void* dst, const void* A, int M, int K, cudaStream_t stream, int pdl = 1);

// Group size along M for the persistent tile order (see gemm_choose_group_m).
int choose_group_m(int M, int N, int K, int tile_m, int tile_n, double bytes_per_row_elem,
                   double extra_bytes_per_row_k, int concurrent_tiles, long long l2_bytes);

}  // namespace dtcp

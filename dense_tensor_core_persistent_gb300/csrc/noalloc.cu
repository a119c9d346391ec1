// noalloc.cu -- gemm_nvfp4_noalloc: the row-major-scale NVFP4 GEMM without any device
// memory allocation.
//
// gemm_nvfp4 needs scratch memory for its scales rearranged into the tensor-core layout,
// and takes it from a stream-ordered memory pool. Some callers cannot let a library
// allocate: code that runs where the CUDA allocator must not be entered (inside a custom
// allocator or memory manager, a signal or error path, a real-time loop that forbids
// allocation latency), or applications that own every byte of device memory through
// their own allocator and account for it. For them this entry point keeps the scratch in
// a fixed array that is part of the library image: it is created when the library's GPU
// code is loaded on a device and stays there until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "gemm.h"
#include "host_common.h"
#include "schedule.h"

namespace dtcp {

// Scratch for the rearranged SFA and SFB of one call (16 MiB; each GPU that loads the
// library holds it until exit). In host code the name is only a host-side stand-in for
// the symbol: the device address comes from cudaGetSymbolAddress below.
constexpr size_t kNoAllocScratchBytes = GEMM_NVFP4_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_noalloc_scale_scratch[kNoAllocScratchBytes];

namespace {

// Device address of the scratch array on `device`, looked up once per device with that
// device current (the caller's current device). nullptr if the lookup fails.
uint8_t* scratch_address(int device) {
  static std::mutex mu;
  static uint8_t* addr[64] = {nullptr};
  if (device < 0 || device >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[device] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scale_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[device] = static_cast<uint8_t*>(p);
  }
  return addr[device];
}

size_t round_up_256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

}  // namespace dtcp

using namespace dtcp;

extern "C" int gemm_nvfp4_noalloc(const void* A, const void* SFA, const void* B, const void* SFB, void* C, int M,
                                  int N, int K, void* stream) {
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_OK;
  if (C == nullptr || (K > 0 && (A == nullptr || B == nullptr || SFA == nullptr || SFB == nullptr)))
    return GEMM_ERR_INVALID_ARG;
  if (K % 256 != 0 || N % 8 != 0 || ceil_div(M, 128) + ceil_div(N, 128) > 65535)
    return GEMM_ERR_UNSUPPORTED_SHAPE;
  if ((reinterpret_cast<uintptr_t>(C) & 15u) != 0 ||
      (K > 0 && ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(SFA) |
                  reinterpret_cast<uintptr_t>(SFB)) & 15u) != 0))
    return GEMM_ERR_MISALIGNED;
  // Both rearranged scale matrices must fit in the fixed scratch array.
  const size_t bytes_a = round_up_256(static_cast<size_t>(ceil_div(M, 128)) * 128 * (static_cast<size_t>(K) / 16));
  const size_t bytes_b = static_cast<size_t>(ceil_div(N, 128)) * 128 * (static_cast<size_t>(K) / 16);
  if (bytes_a + bytes_b > kNoAllocScratchBytes) return GEMM_ERR_SCRATCH_TOO_SMALL;
  // Few rows: A is read from a copy padded to 32 rows (as gemm_nvfp4 does), placed after the
  // scales when the array has room for it; otherwise A is read in place.
  const RunOptions opt;
  int a_rows = nvfp4_a_rows(M, opt);
  const size_t off_pad = round_up_256(bytes_a + bytes_b);
  if (a_rows != M && off_pad + static_cast<size_t>(a_rows) * (static_cast<size_t>(K) / 2) > kNoAllocScratchBytes)
    a_rows = M;
  int device = 0, err = 0;
  if (current_device_info(&device, &err) == nullptr) return err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) {
    if (cudaMemsetAsync(C, 0, size_t(M) * size_t(N) * 2, s) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
  }
  uint8_t* scratch = scratch_address(device);
  if (scratch == nullptr) return GEMM_ERR_NO_DEVICE;
  // The pack kernel writes every byte the GEMM reads (padding rows as zeros), so nothing
  // left in the array by an earlier call needs clearing. (The rows of the padded A past M
  // keep an earlier call's bytes: they only reach C rows that are never stored.)
  uint8_t* a_pad = a_rows != M ? scratch + off_pad : nullptr;
  int st = run_pack_scales2_copy(SFA, scratch, M, SFB, scratch + bytes_a, N, K, A, a_pad,
                                 a_pad ? static_cast<long long>(M) * (K / 2) : 0, s);
  const void* a_src = a_pad ? a_pad : A;
  if (st == GEMM_OK) st = run_gemm_nvfp4_blocked(a_src, scratch, B, scratch + bytes_a, C, M, N, K, s, opt, a_rows);
  return st;
}

// api.cu -- the extern "C" entry points declared in include/gemm.h: argument validation,
// device facts, tensor-map encoding (cuTensorMapEncodeTiled through the runtime's driver
// entry point, so the library needs no -lcuda), the device status word, and the host
// helpers for the tile order.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "gemm.h"
#include "host_common.h"
#include "schedule.h"

namespace dtcp {

// ---------------------------------------------------------------- status word

// One word per device (a static __device__ variable: nothing is allocated). Kernels
// store the first error they hit; gemm_get_device_status reads and clears it.
__device__ unsigned g_status_word;

unsigned* device_status_word(int device) {
  static std::mutex mu;
  static unsigned* addr[64] = {nullptr};
  if (device < 0 || device >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[device] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[device] = static_cast<unsigned*>(p);
  }
  return addr[device];
}

// ---------------------------------------------------------------- device facts

const DeviceInfo* current_device_info(int* device, int* err) {
  static std::mutex mu;
  static DeviceInfo infos[64];
  static bool have[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    *err = GEMM_ERR_NO_DEVICE;
    return nullptr;
  }
  *device = dev;
  std::lock_guard<std::mutex> lock(mu);
  if (!have[dev]) {
    DeviceInfo d;
    int l2 = 0;
    if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
      cudaGetLastError();
      *err = GEMM_ERR_NO_DEVICE;
      return nullptr;
    }
    d.l2_bytes = l2;
    infos[dev] = d;
    have[dev] = true;
  }
  const DeviceInfo* d = &infos[dev];
  // The kernels are built for sm_103a only (tcgen05, CTA pairs, 227 KB of shared memory).
  if (d->cc_major != 10 || d->cc_minor != 3) {
    *err = GEMM_ERR_ARCH;
    return nullptr;
  }
  return d;
}

// ---------------------------------------------------------------- tensor maps

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

std::atomic<unsigned long long> g_launches{0};

}  // namespace

// Encoded tensor maps of recent calls, per host thread: a map depends only on the
// parameters in its key (address, type, sizes, strides, box, swizzle), so a repeated call
// reuses it instead of encoding again (each encode costs the host about half a microsecond,
// and a call needs up to five).
namespace {
struct TmapKey {
  const void* base;
  int rank, dtype, swizzle, pad;
  uint64_t dims[3];
  uint64_t strides[2];
  uint32_t box[3], pad2;
};
struct TmapEntry {
  TmapKey key;
  CUtensorMap map;
  bool valid;
};
constexpr int kTmapCacheEntries = 32;
thread_local TmapEntry t_tmap_cache[kTmapCacheEntries];
thread_local int t_tmap_next = 0;

int encode_cached(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
                  const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  TmapKey key;
  std::memset(&key, 0, sizeof(key));  // padding included: keys compare with memcmp
  key.base = base;
  key.rank = rank;
  key.dtype = static_cast<int>(dtype);
  key.swizzle = static_cast<int>(swizzle);
  for (int i = 0; i < rank; ++i) key.dims[i] = dims[i];
  for (int i = 0; i + 1 < rank; ++i) key.strides[i] = strides_bytes[i];
  for (int i = 0; i < rank; ++i) key.box[i] = box[i];
  for (TmapEntry& e : t_tmap_cache)
    if (e.valid && std::memcmp(&e.key, &key, sizeof(key)) == 0) {
      *map = e.map;
      return GEMM_OK;
    }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return GEMM_ERR_DRIVER;
  cuuint64_t d[3], st[2];
  cuuint32_t b[3];
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) st[i] = strides_bytes[i];
  // Out-of-bounds elements of a load are filled with zeros ("NONE" = no NaN request),
  // which leaves every sum unchanged; out-of-bounds elements of a store are dropped.
  const CUresult r = fn(map, dtype, rank, const_cast<void*>(base), d, st, b, elem_strides,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return GEMM_ERR_DRIVER;
  TmapEntry& slot = t_tmap_cache[t_tmap_next];
  t_tmap_next = (t_tmap_next + 1) % kTmapCacheEntries;
  slot.key = key;
  slot.map = *map;
  slot.valid = true;
  return GEMM_OK;
}
}  // namespace

int encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner_elems,
                   uint64_t outer_rows, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                   CUtensorMapSwizzle swizzle) {
  const uint64_t dims[2] = {inner_elems, outer_rows};
  const uint64_t strides[1] = {row_stride_bytes};
  const uint32_t box[2] = {box_inner, box_outer};
  return encode_cached(map, dtype, 2, base, dims, strides, box, swizzle);
}

int encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, const uint64_t dims[3],
                   const uint64_t strides_bytes[2], const uint32_t box[3], CUtensorMapSwizzle swizzle) {
  return encode_cached(map, dtype, 3, base, dims, strides_bytes, box, swizzle);
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// ---------------------------------------------------------------- tile order

int choose_group_m(int M, int N, int K, int tile_m, int tile_n, double bytes_per_row_elem,
                   double extra_bytes_per_row_k, int concurrent_tiles, long long l2_bytes) {
  const int num_m = ceil_div(M, tile_m);
  const int num_n = ceil_div(N, tile_n);
  if (num_m <= 1 || num_n <= 1) return std::max(num_m, 1);
  const double per_k = bytes_per_row_elem + extra_bytes_per_row_k;
  const double a_total = double(M) * K * per_k, b_total = double(N) * K * per_k;
  // Both operands fit in L2: any order re-reads from L2 only; walk all of M per column.
  if (a_total + b_total <= double(l2_bytes)) return num_m;
  // Bytes of one A tile and one B tile over the whole K.
  const double w_a = double(tile_m) * K * per_k, w_b = double(tile_n) * K * per_k;
  // Two waves of tiles share L2: every other wave walks K downwards and starts on the K
  // blocks the previous one read last. (Measured on GB300, BF16: the two-wave group 12 in
  // place of the one-wave 9 gained 0.8% at 8192^3, 1.0% at 6144^3, 0.2% at 4000 x 14336 x 4096.)
  const int c = 2 * std::max(concurrent_tiles, 1);
  // c consecutive tiles touch g A tiles and about c/g B tiles; equal bytes of A and B
  // (the smallest footprint) at g = sqrt(c * w_b / w_a).
  int g = static_cast<int>(std::lround(std::sqrt(double(c) * w_b / w_a)));
  g = std::min(std::max(g, 1), num_m);
  auto footprint = [&](int gg) { return gg * w_a + std::ceil(double(c) / gg) * w_b; };
  // Shrink while the two waves' operands do not fit in L2 and a smaller group still has a
  // smaller footprint (the rounding of the square root may leave it one step off the
  // smallest). Once nothing fits, the balanced group still re-reads least: each wave reads
  // g A tiles and c/g B tiles per K block from DRAM, with no reuse across waves either way.
  while (g > 1 && footprint(g) > double(l2_bytes) && footprint(g - 1) < footprint(g)) --g;
  return g;
}

// ---------------------------------------------------------------- validation helpers

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int resolve_options(const gemm_options_t* o, RunOptions* r) {
  if (o == nullptr) return GEMM_OK;
  if (o->clc < 0 || o->clc > 2) return GEMM_ERR_INVALID_ARG;
  if (o->no_swap_ab != 0 && o->no_swap_ab != 1) return GEMM_ERR_INVALID_ARG;
  if (o->no_split_k != 0 && o->no_split_k != 1) return GEMM_ERR_INVALID_ARG;
  if (o->no_tail_split != 0 && o->no_tail_split != 1) return GEMM_ERR_INVALID_ARG;
  if (o->no_pdl != 0 && o->no_pdl != 1) return GEMM_ERR_INVALID_ARG;
  if (o->no_pad_a != 0 && o->no_pad_a != 1) return GEMM_ERR_INVALID_ARG;
  if (o->clock_probe_ctas < 0 || (o->clock_probe_ctas > 0 && o->clock_probe == nullptr)) return GEMM_ERR_INVALID_ARG;
  if (o->kernel < GEMM_KERNEL_DEFAULT || o->kernel > GEMM_KERNEL_BF16_2CTA_WIDE) return GEMM_ERR_INVALID_ARG;
  if (o->group_m < 0 || o->max_clusters < 0 || (o->persistent != 0 && o->persistent != 1))
    return GEMM_ERR_INVALID_ARG;
  if (o->debug_flags & ~1u) return GEMM_ERR_INVALID_ARG;
  r->kernel = o->kernel;
  r->persistent = o->persistent;
  r->group_m = o->group_m;
  r->max_clusters = o->max_clusters;
  r->tail_split = o->no_tail_split ? 0 : 1;
  r->pdl = o->no_pdl ? 0 : 1;
  r->swap_ab = o->no_swap_ab ? 0 : 1;
  r->split_k = o->no_split_k ? 0 : 1;
  r->clc = o->clc;
  r->pad_a = o->no_pad_a ? 0 : 1;
  r->clock_probe = o->clock_probe_ctas > 0 ? o->clock_probe : nullptr;
  r->clock_probe_ctas = o->clock_probe_ctas;
  if (o->wait_limit_us != 0) r->wait_limit_ns = uint64_t(o->wait_limit_us) * 1000ull;
  r->debug_flags = o->debug_flags;
  return GEMM_OK;
}

static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// A stream-ordered memory pool owned by the library, one per device, for the temporary
// blocked-scale workspace of gemm_nvfp4. Freed blocks stay in the pool (release threshold
// at the maximum), so after the first calls the workspace costs no allocation from the
// driver; blocks freed on one stream are reused by later work on any stream in order.
cudaMemPool_t workspace_pool(int device) {
  static std::mutex mu;
  static cudaMemPool_t pools[64] = {nullptr};
  if (device < 0 || device >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (pools[device] == nullptr) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = device;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    uint64_t keep = ~0ull;
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    pools[device] = pool;
  }
  return pools[device];
}

// C = 0 for an empty K (the sum over no terms); BF16 zero is the all-zero bit pattern.
static int zero_output(void* C, int M, int N, cudaStream_t stream) {
  if (cudaMemsetAsync(C, 0, size_t(M) * size_t(N) * 2, stream) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

// Checks a gemm_epilogue_t; NULL is the identity.
static int resolve_epilogue(const gemm_epilogue_t* e, EpilogueOptions* r) {
  if (e == nullptr) return GEMM_OK;
  if (e->reserved != 0) return GEMM_ERR_INVALID_ARG;
  if (e->activation != GEMM_ACT_NONE && e->activation != GEMM_ACT_RELU && e->activation != GEMM_ACT_GELU_TANH)
    return GEMM_ERR_INVALID_ARG;
  if (e->bias != nullptr && !aligned16(e->bias)) return GEMM_ERR_MISALIGNED;
  r->alpha = e->alpha;
  r->beta = e->beta;
  r->bias = e->bias;
  r->act = e->activation;
  return GEMM_OK;
}

// K == 0 with a fused epilogue: the product is zero, so C = act(beta * C + bias), 8
// elements (one 16-byte vector; N is a multiple of 8) per thread and step.
__global__ void epilogue_only_kernel(uint16_t* C, long long vectors, int N, EpiParams e) {
  for (long long v = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; v < vectors;
       v += static_cast<long long>(gridDim.x) * blockDim.x) {
    uint4* c = reinterpret_cast<uint4*>(C) + v;
    const int col = static_cast<int>((v * 8) % N);
    const uint4 old = e.beta != 0.0f ? *c : make_uint4(0u, 0u, 0u, 0u);  // beta == 0: C is not read
    const uint4 b = epi_bias8(e, col, N);
    *c = make_uint4(epi_pair(0u, 0u, old.x, b.x, e), epi_pair(0u, 0u, old.y, b.y, e), epi_pair(0u, 0u, old.z, b.z, e),
                    epi_pair(0u, 0u, old.w, b.w, e));
  }
}

static int empty_sum_output(void* C, int M, int N, cudaStream_t stream, const EpilogueOptions& epi, int num_sms) {
  if (!epi.fused()) return zero_output(C, M, N, stream);
  EpiParams e;
  e.alpha = epi.alpha;
  e.beta = epi.beta;
  e.bias = static_cast<const uint16_t*>(epi.bias);
  e.act = epi.act;
  e.fused = 1;
  const long long vectors = static_cast<long long>(M) * N / 8;
  const long long want = (vectors + 255) / 256;
  const int blocks = static_cast<int>(std::min<long long>(want, 8LL * std::max(num_sms, 1)));
  epilogue_only_kernel<<<blocks, 256, 0, stream>>>(static_cast<uint16_t*>(C), vectors, N, e);
  if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_LAUNCH;
  count_launch();
  return GEMM_OK;
}

}  // namespace dtcp

using namespace dtcp;

extern "C" {

int gemm_bf16_fused(const void* A, const void* B, void* C, int M, int N, int K, void* stream,
                    const gemm_epilogue_t* epilogue, const gemm_options_t* options) {
  RunOptions opt;
  int st = resolve_options(options, &opt);
  if (st == GEMM_OK) st = resolve_epilogue(epilogue, &opt.epi);
  if (st != GEMM_OK) return st;
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_OK;
  if (C == nullptr || (K > 0 && (A == nullptr || B == nullptr))) return GEMM_ERR_INVALID_ARG;
  if (K % 8 != 0 || N % 8 != 0) return GEMM_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(C) || (K > 0 && (!aligned16(A) || !aligned16(B)))) return GEMM_ERR_MISALIGNED;
  int device = 0, err = 0;
  const DeviceInfo* info = current_device_info(&device, &err);
  if (info == nullptr) return err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return empty_sum_output(C, M, N, s, opt.epi, info->num_sms);
  return run_gemm_bf16(A, B, C, M, N, K, s, opt);
}

int gemm_bf16_ex(const void* A, const void* B, void* C, int M, int N, int K, void* stream,
                 const gemm_options_t* options) {
  return gemm_bf16_fused(A, B, C, M, N, K, stream, nullptr, options);
}

int gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K, void* stream) {
  return gemm_bf16_ex(A, B, C, M, N, K, stream, nullptr);
}

int gemm_nvfp4_fused(const void* A, const void* SFA, const void* B, const void* SFB, void* C, int M, int N, int K,
                     void* stream, const gemm_epilogue_t* epilogue, const gemm_options_t* options) {
  RunOptions opt;
  int st = resolve_options(options, &opt);
  if (st == GEMM_OK) st = resolve_epilogue(epilogue, &opt.epi);
  if (st != GEMM_OK) return st;
  if (opt.kernel != GEMM_KERNEL_DEFAULT) return GEMM_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_OK;
  if (C == nullptr || (K > 0 && (A == nullptr || B == nullptr || SFA == nullptr || SFB == nullptr)))
    return GEMM_ERR_INVALID_ARG;
  if (K % 256 != 0 || N % 8 != 0 || ceil_div(M, 128) + ceil_div(N, 128) > 65535)
    return GEMM_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(C) || (K > 0 && (!aligned16(A) || !aligned16(B) || !aligned16(SFA) || !aligned16(SFB))))
    return GEMM_ERR_MISALIGNED;
  int device = 0, err = 0;
  const DeviceInfo* info = current_device_info(&device, &err);
  if (info == nullptr) return err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return empty_sum_output(C, M, N, s, opt.epi, info->num_sms);
  // Rearrange both scale matrices into the blocked layout in a stream-ordered workspace
  // (and, for few rows, copy A into a padded buffer there), run the blocked GEMM, and free
  // the workspace in stream order behind it.
  const size_t bytes_a = round_up(static_cast<size_t>(gemm_nvfp4_blocked_scale_bytes(M, K)), 256);
  const size_t bytes_b = round_up(static_cast<size_t>(gemm_nvfp4_blocked_scale_bytes(N, K)), 256);
  const int a_rows = nvfp4_a_rows(M, opt);
  const size_t bytes_pad = a_rows != M ? static_cast<size_t>(a_rows) * (static_cast<size_t>(K) / 2) : 0;
  cudaMemPool_t pool = workspace_pool(device);
  void* ws = nullptr;
  if (pool == nullptr || cudaMallocFromPoolAsync(&ws, bytes_a + bytes_b + bytes_pad, pool, s) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_OUT_OF_MEMORY;
  }
  uint8_t* sfa_blk = static_cast<uint8_t*>(ws);
  uint8_t* sfb_blk = sfa_blk + bytes_a;
  // (few rows: the packing launch also copies A's rows into the padded buffer)
  uint8_t* a_pad = bytes_pad > 0 ? sfb_blk + bytes_b : nullptr;
  st = run_pack_scales2_copy(SFA, sfa_blk, M, SFB, sfb_blk, N, K, A, a_pad,
                             a_pad ? static_cast<long long>(M) * (K / 2) : 0, s, opt.pdl);
  const void* a_src = a_pad ? a_pad : A;
  if (st == GEMM_OK) st = run_gemm_nvfp4_blocked(a_src, sfa_blk, B, sfb_blk, C, M, N, K, s, opt, a_rows);
  if (cudaFreeAsync(ws, s) != cudaSuccess && st == GEMM_OK) st = GEMM_ERR_LAUNCH;
  return st;
}

int gemm_nvfp4_ex(const void* A, const void* SFA, const void* B, const void* SFB, void* C, int M, int N, int K,
                  void* stream, const gemm_options_t* options) {
  return gemm_nvfp4_fused(A, SFA, B, SFB, C, M, N, K, stream, nullptr, options);
}

int gemm_nvfp4(const void* A, const void* SFA, const void* B, const void* SFB, void* C, int M, int N, int K,
               void* stream) {
  return gemm_nvfp4_ex(A, SFA, B, SFB, C, M, N, K, stream, nullptr);
}

long long gemm_nvfp4_blocked_scale_bytes(int rows, int K) {
  if (rows < 0 || K < 0 || K % 64 != 0) return -1;
  return static_cast<long long>(ceil_div(rows, 128)) * 128 * (K / 16);
}

int gemm_nvfp4_pack_scales(const void* SF, void* SF_blocked, int rows, int K, void* stream) {
  if (rows < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  if (K % 64 != 0 || ceil_div(rows, 128) > 65535) return GEMM_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0 || K == 0) return GEMM_OK;
  if (SF == nullptr || SF_blocked == nullptr) return GEMM_ERR_INVALID_ARG;
  if (!aligned16(SF) || !aligned16(SF_blocked)) return GEMM_ERR_MISALIGNED;
  int device = 0, err = 0;
  if (current_device_info(&device, &err) == nullptr) return err;
  return run_pack_scales(SF, SF_blocked, rows, K, static_cast<cudaStream_t>(stream));
}

int gemm_nvfp4_blocked_fused(const void* A, const void* SFA_blocked, const void* B, const void* SFB_blocked, void* C,
                             int M, int N, int K, void* stream, const gemm_epilogue_t* epilogue,
                             const gemm_options_t* options) {
  RunOptions opt;
  int st = resolve_options(options, &opt);
  if (st == GEMM_OK) st = resolve_epilogue(epilogue, &opt.epi);
  if (st != GEMM_OK) return st;
  if (opt.kernel != GEMM_KERNEL_DEFAULT) return GEMM_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_OK;
  if (C == nullptr || (K > 0 && (A == nullptr || B == nullptr || SFA_blocked == nullptr || SFB_blocked == nullptr)))
    return GEMM_ERR_INVALID_ARG;
  if (K % 256 != 0 || N % 8 != 0) return GEMM_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(C) ||
      (K > 0 && (!aligned16(A) || !aligned16(B) || !aligned16(SFA_blocked) || !aligned16(SFB_blocked))))
    return GEMM_ERR_MISALIGNED;
  int device = 0, err = 0;
  const DeviceInfo* info = current_device_info(&device, &err);
  if (info == nullptr) return err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return empty_sum_output(C, M, N, s, opt.epi, info->num_sms);
  const int a_rows = nvfp4_a_rows(M, opt);
  if (a_rows == M) return run_gemm_nvfp4_blocked(A, SFA_blocked, B, SFB_blocked, C, M, N, K, s, opt);
  // few rows: A from a padded copy in a stream-ordered workspace, freed in order behind the GEMM
  cudaMemPool_t pool = workspace_pool(device);
  void* ws = nullptr;
  if (pool == nullptr ||
      cudaMallocFromPoolAsync(&ws, static_cast<size_t>(a_rows) * (static_cast<size_t>(K) / 2), pool, s) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_OUT_OF_MEMORY;
  }
  st = run_copy_rows(ws, A, M, K, s, opt.pdl);
  if (st == GEMM_OK) st = run_gemm_nvfp4_blocked(ws, SFA_blocked, B, SFB_blocked, C, M, N, K, s, opt, a_rows);
  if (cudaFreeAsync(ws, s) != cudaSuccess && st == GEMM_OK) st = GEMM_ERR_LAUNCH;
  return st;
}

int gemm_nvfp4_blocked_ex(const void* A, const void* SFA_blocked, const void* B, const void* SFB_blocked, void* C,
                          int M, int N, int K, void* stream, const gemm_options_t* options) {
  return gemm_nvfp4_blocked_fused(A, SFA_blocked, B, SFB_blocked, C, M, N, K, stream, nullptr, options);
}

int gemm_nvfp4_blocked(const void* A, const void* SFA_blocked, const void* B, const void* SFB_blocked, void* C, int M,
                       int N, int K, void* stream) {
  return gemm_nvfp4_blocked_ex(A, SFA_blocked, B, SFB_blocked, C, M, N, K, stream, nullptr);
}

int gemm_bf16_plan(int M, int N, int K, const gemm_options_t* options, const gemm_epilogue_t* epilogue, int* swap_ab,
                   int* tile_n) {
  if (M < 0 || N < 0 || K < 0 || swap_ab == nullptr || tile_n == nullptr) return GEMM_ERR_INVALID_ARG;
  RunOptions opt;
  int st = resolve_options(options, &opt);
  if (st == GEMM_OK) st = resolve_epilogue(epilogue, &opt.epi);
  if (st != GEMM_OK) return st;
  *swap_ab = bf16_swap_ab(M, N, opt) ? 1 : 0;
  *tile_n = bf16_tile_n(M, N, opt);
  return GEMM_OK;
}

int gemm_nvfp4_plan(int M, int N, int K, const gemm_options_t* options, int* a_rows) {
  RunOptions opt;
  if (resolve_options(options, &opt) != GEMM_OK || a_rows == nullptr || M < 0 || N < 0 || K < 0)
    return GEMM_ERR_INVALID_ARG;
  *a_rows = nvfp4_a_rows(M, opt);
  return GEMM_OK;
}

const char* gemm_status_string(int status) {
  switch (status) {
    case GEMM_OK: return "ok";
    case GEMM_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case GEMM_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case GEMM_ERR_NO_DEVICE: return "no CUDA device";
    case GEMM_ERR_ARCH: return "device is not sm_103 (GB300)";
    case GEMM_ERR_DRIVER: return "tensor map encoding failed";
    case GEMM_ERR_LAUNCH: return "kernel launch failed";
    case GEMM_ERR_TIMEOUT: return "device wait timed out";
    case GEMM_ERR_OUT_OF_MEMORY: return "out of device memory for the scale workspace";
    case GEMM_ERR_SCRATCH_TOO_SMALL:
      return "problem's rearranged scales exceed the fixed no-allocation scratch array (16 MiB)";
    default: return "unknown status";
  }
}

int gemm_get_device_status(void* stream, uint32_t* detail) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  unsigned word = 0;
  const unsigned zero = 0;
  if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  if (detail) *detail = word;
  return static_cast<int>(word & 0xFFu);
}

int gemm_tile_coord(int M, int N, int tile_m, int tile_n, int group_m, int t, int* m_blk, int* n_blk) {
  if (M <= 0 || N <= 0 || tile_m <= 0 || tile_n <= 0 || group_m <= 0 || m_blk == nullptr || n_blk == nullptr)
    return GEMM_ERR_INVALID_ARG;
  const int num_m = ceil_div(M, tile_m), num_n = ceil_div(N, tile_n);
  if (t < 0 || static_cast<long long>(t) >= static_cast<long long>(num_m) * num_n) return GEMM_ERR_INVALID_ARG;
  const TileCoord c = tile_coord(t, num_m, num_n, group_m);
  *m_blk = c.m_blk;
  *n_blk = c.n_blk;
  return GEMM_OK;
}

int gemm_choose_group_m(int M, int N, int K, int tile_m, int tile_n, int elem_bytes_x2, int concurrent_tiles,
                        long long l2_bytes) {
  if (M <= 0 || N <= 0 || K <= 0 || tile_m <= 0 || tile_n <= 0 || elem_bytes_x2 <= 0 || l2_bytes <= 0)
    return -GEMM_ERR_INVALID_ARG;
  // elem_bytes_x2 == 1 means packed E2M1 (half a byte) plus one scale byte per 16 elements.
  const double per = elem_bytes_x2 * 0.5;
  const double extra = (elem_bytes_x2 == 1) ? 1.0 / 16.0 : 0.0;
  return choose_group_m(M, N, K, tile_m, tile_n, per, extra, concurrent_tiles, l2_bytes);
}

int gemm_clc_rule(int items, int wave, int K, int nvfp4) {
  if (items < 0 || wave <= 0 || K < 0 || (nvfp4 != 0 && nvfp4 != 1)) return -GEMM_ERR_INVALID_ARG;
  return clc_rule(items, wave, K, nvfp4 != 0) ? 1 : 0;
}

int gemm_bf16_wide_rule(int M, int N, int K, int wave) {
  if (M < 0 || N < 0 || K < 0 || wave <= 0) return -GEMM_ERR_INVALID_ARG;
  return wide_rule(M, N, K, wave) ? 1 : 0;
}

unsigned long long gemm_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"

// common.cuh -- pieces shared by the BF16 and NVFP4 kernels: tcgen05 descriptors,
// bounded mbarrier waits with error reporting, and the status-word layout.
#pragma once

#include <cstdint>

#include "ptx.cuh"
#include "schedule.h"

namespace dtcp {

// Error word written by kernels: bits 0-7 status code, 8-15 role, 16-31 stage/slot.
constexpr uint32_t kStatusTimeout = 8;  // == GEMM_ERR_TIMEOUT
enum Role : uint32_t { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3, kRoleScales = 4 };

__host__ __device__ constexpr uint32_t status_code(uint32_t role, uint32_t index) {
  return kStatusTimeout | (role << 8) | (index << 16);
}

// ---------------------------------------------------------------- descriptors

// Shared-memory matrix descriptor (tcgen05 / sm_100 family) for a K-major operand tile
// written by TMA with 128-byte swizzle: every row is 128 bytes of K, eight rows form a
// 1024-byte swizzle atom, atoms are stacked along M (or N) 1024 bytes apart. The tile
// must start on a 1024-byte boundary; a K offset inside the 128-byte row is applied by
// adding it to the start address (the swizzle is a function of the address bits).
// ("Achieve cuBLAS Performance on NVIDIA GB300 for HGEMM", v1: the MMA descriptor
// selects the 128-byte swizzle mode, 2 << 61, so the TMA-written layout and the
// MMA-read layout coincide.)
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
  return static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu)  // bits 0-13: start address / 16
         | (static_cast<uint64_t>(1) << 16)                 // bits 16-29: leading offset (unused here)
         | (static_cast<uint64_t>(1024 >> 4) << 32)         // bits 32-45: stride between 8-row atoms / 16
         | (static_cast<uint64_t>(1) << 46)                 // bits 46-47: descriptor version 1
         | (static_cast<uint64_t>(2) << 61);                // bits 61-63: 128-byte swizzle
}

// Descriptor of an unswizzled source made of 8-row x 16-byte core matrices with the
// rows of a core matrix contiguous (16 bytes apart) and successive core matrices along
// the row dimension `sbo_bytes` apart.
__device__ __forceinline__ uint64_t umma_desc_plain(uint32_t smem_addr, uint32_t sbo_bytes) {
  return static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(0) << 16) |
         (static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46);
}

// Descriptor of the operand `bytes` further on (bytes % 16 == 0): the start address is the
// low field, and shared-memory addresses stay below 2^18, so the field never overflows.
__device__ __forceinline__ uint64_t umma_desc_advance(uint64_t desc, uint32_t bytes) {
  return desc + static_cast<uint64_t>(bytes >> 4);
}

// Instruction descriptor, kind::f16: BF16 x BF16 -> FP32, both operands K-major.
// bits 4-5 D format (1 = F32), 7-9 A format (1 = BF16), 10-12 B format (1 = BF16),
// 15/16 A/B major (0 = K), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// Instruction descriptor, kind::mxf4nvf4 block-scaled: E2M1 x E2M1 -> FP32 with UE4M3
// scale factors (bit 23 = 0), both operands K-major; scale-factor ids 0 (bits 4-5, 29-30).
// bits 7-9 / 10-12 A / B format (1 = E2M1), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_nvf4(int m, int n) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// ---------------------------------------------------------------- bounded waits

struct WaitCtx {
  volatile uint32_t* abort_flag;  // this CTA's shared abort flag
  unsigned* status;               // device status word
  uint64_t limit_ns;              // bound on one wait
};

static __device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, WaitCtx w, uint32_t code,
                                             bool honour_abort) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    // suspended waits of at most 20 us, so the abort flag and the time limit are
    // still checked often; a completed phase wakes the thread at once
    if (mbar_try_wait_suspend(bar, parity, 20000u)) return true;
    if (honour_abort && *w.abort_flag) return false;
    if (globaltimer_ns() - t0 > w.limit_ns) {
      atomicCAS(w.status, 0u, code);
      *w.abort_flag = 1u;
      return false;
    }
  }
}

// Wait until the phase with parity `parity` of `bar` has completed. Returns false if
// the wait gave up: after `limit_ns` (the error `code` is recorded in the status word
// and this CTA's abort flag is raised) or because another role of this CTA aborted.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const WaitCtx& w, uint32_t code) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_phase_slow(bar, parity, w, code, true);
}

// Same wait with the slow path inlined: for code that runs under a changed register
// limit (setmaxnreg), where a call to an out-of-line function is not allowed to follow
// the caller's register budget.
__device__ __forceinline__ bool wait_phase_inline(uint32_t bar, uint32_t parity, const WaitCtx& w, uint32_t code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_suspend(bar, parity, 20000u)) return true;
    if (*w.abort_flag) return false;
    if (globaltimer_ns() - t0 > w.limit_ns) {
      atomicCAS(w.status, 0u, code);
      *w.abort_flag = 1u;
      return false;
    }
  }
}

// Warp-collective form: every lane waits (so every lane acquires what the barrier
// guards), and the outcome is made uniform so the warp leaves its loop together.
__device__ __forceinline__ bool wait_phase_warp(uint32_t bar, uint32_t parity, const WaitCtx& w, uint32_t code) {
  const bool ok = wait_phase(bar, parity, w, code);
  return __all_sync(0xffffffffu, ok) != 0;
}

// After an abort: give copies this thread started time to land before the CTA exits.
__device__ __forceinline__ void settle_after_abort() {
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < 1000000ull) __nanosleep(1000);
}

// ---------------------------------------------------------------- work-item sequence

// A cluster computes a sequence of work items. Static scheduling: its own cluster index,
// then steps of the number of launched clusters. Cluster launch control (CLC): the grid
// has one cluster per item; a running cluster starts on its own index and then takes the
// item of each cluster it cancels before that cluster starts ("NVFP4 GEMM on Blackwell",
// Kernel 5: the full logical grid is launched and each resident cluster cancels a pending
// one and takes its tile). Response t of a ring of kClcSlots 16-byte slots names the
// item after item t of the sequence.
//
// One thread of the leader CTA requests response t when it starts item t (once every
// consumer has released response t - kClcSlots from that slot); the response is written
// to both CTAs of a pair. Every role that walks the items reads response t when it is
// done with item t; in each CTA the thread that arms full[s] re-arms it for the next use
// of the slot, and the others release the slot on the leader's empty[s].
constexpr int kClcSlots = 4;

struct ClcRing {
  uint32_t resp;          // this CTA's response slot 0 (slot s at resp + 16 s)
  uint32_t full;          // this CTA's full[0] (armed with 16 transaction bytes per use)
  uint32_t empty_leader;  // the leader CTA's empty[0], as a shared::cluster address
};

// INLINE: the waits are inlined (for roles running under a changed register limit).
template <bool INLINE>
__device__ __forceinline__ bool clc_wait(uint32_t bar, uint32_t parity, const WaitCtx& w, uint32_t code) {
  if constexpr (INLINE) return wait_phase_inline(bar, parity, w, code);
  else return wait_phase(bar, parity, w, code);
}

// Issuer: request response t (the item after this cluster's item t).
template <bool MULTICAST, bool INLINE = false>
__device__ __forceinline__ bool clc_request(const ClcRing& r, uint32_t empty_local, int t, const WaitCtx& w,
                                            uint32_t code) {
  const uint32_t s = static_cast<uint32_t>(t) % kClcSlots, ph = (static_cast<uint32_t>(t) / kClcSlots) & 1u;
  if (!clc_wait<INLINE>(empty_local + 8 * s, ph ^ 1u, w, code)) return false;
  fence_proxy_async_smem();  // the consumers' reads of the slot before its next asynchronous write
  clc_try_cancel<MULTICAST>(r.resp + 16 * s, r.full + 8 * s);
  return true;
}

// Response t of the slot ring: the next item (the cancelled cluster's first CTA index /
// cg), or -1 when no cluster was left to cancel or the wait gave up (then ok = false).
// `arm`: this thread re-arms full[s] for the slot's next use; `release`: it arrives on
// the leader's empty[s] (every consumer but the issuer).
template <bool INLINE = false>
__device__ __forceinline__ int clc_next(const ClcRing& r, int t, int cg, bool arm, bool release, const WaitCtx& w,
                                        uint32_t code, bool& ok) {
  const uint32_t s = static_cast<uint32_t>(t) % kClcSlots, ph = (static_cast<uint32_t>(t) / kClcSlots) & 1u;
  if (!clc_wait<INLINE>(r.full + 8 * s, ph, w, code)) {
    ok = false;
    return -1;
  }
  uint32_t x;
  const bool got = clc_query(r.resp + 16 * s, x);
  if (got && arm) mbar_arrive_expect_tx(r.full + 8 * s, 16);
  if (release) mbar_arrive_cluster_relaxed(r.empty_leader + 8 * s);
  return got ? static_cast<int>(x) / cg : -1;
}

// ---------------------------------------------------------------- clock probe

// gemm_options_t.clock_probe: thread 0 of each CTA (blockIdx.x < ctas) stores %globaltimer
// and the SM's clock64 when its work starts (after the dependency wait, slot 0) and when
// it ends (after the teardown barrier, slot 1): buf[4 b + 2 slot] and buf[4 b + 2 slot + 1].
// The ratio of the differences is the SM clock the CTA ran at. Null buf: nothing is stored.
struct ClockProbe {
  unsigned long long* buf;
  int ctas;
};
__device__ __forceinline__ void clock_probe_mark(const ClockProbe& c, int slot) {
  if (c.buf != nullptr && threadIdx.x == 0 && static_cast<int>(blockIdx.x) < c.ctas) {
    c.buf[4 * blockIdx.x + 2 * slot] = globaltimer_ns();
    c.buf[4 * blockIdx.x + 2 * slot + 1] = static_cast<unsigned long long>(clock64());
  }
}

// ---------------------------------------------------------------- fused epilogue

// C = act(alpha * acc + beta * C_old + bias[col]), in FP32, rounded once to BF16.
// `fused` is 0 for the plain epilogue (alpha 1, beta 0, no bias, no activation).
struct EpiParams {
  float alpha, beta;
  const uint16_t* bias;  // N BF16 values, or null
  int act;               // 0 none, 1 ReLU, 2 GELU (tanh form)
  int fused;
};

// Two FP32 values in one 64-bit register: the packed forms of mul, fma and add (.f32x2)
// handle a pair of adjacent columns in one instruction.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float r;  // rcp.approx of +inf is 0
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// One pair of adjacent columns: FP32 accumulator bits acc0 / acc1, the prior C and the
// bias as BF16 pairs (element 0 in the low half). x = alpha * acc + beta * C_old + bias,
// then the activation, then one rounding to BF16.
__device__ __forceinline__ uint32_t epi_pair(uint32_t acc0, uint32_t acc1, uint32_t old2, uint32_t bias2,
                                             const EpiParams& e) {
  uint64_t x = f2_mul(f2_pack(e.alpha, e.alpha), f2_pack(__uint_as_float(acc0), __uint_as_float(acc1)));
  if (e.beta != 0.0f)
    x = f2_fma(f2_pack(e.beta, e.beta), f2_pack(__uint_as_float(old2 << 16), __uint_as_float(old2 & 0xFFFF0000u)), x);
  x = f2_add(x, f2_pack(__uint_as_float(bias2 << 16), __uint_as_float(bias2 & 0xFFFF0000u)));
  float y0, y1;
  if (e.act == 2) {
    // GELU, tanh form: 0.5 x (1 + tanh(u)), u = sqrt(2/pi) (x + 0.044715 x^3), evaluated as
    // x / (1 + exp(-2u)) (the same function: 0.5 (1 + tanh u) is the logistic function of
    // 2u); exp(-2u) = 2^(t * -2 sqrt(2/pi) / ln 2) with t = x + 0.044715 x^3. If the power
    // overflows, 1 / inf = 0 and the result is -0.
    const uint64_t t = f2_fma(f2_mul(x, f2_pack(0.044715f, 0.044715f)), f2_mul(x, x), x);
    float v0, v1;
    f2_unpack(f2_mul(t, f2_pack(-2.302208198144325f, -2.302208198144325f)), v0, v1);
    float d0, d1;
    f2_unpack(f2_add(f2_pack(ex2_approx(v0), ex2_approx(v1)), f2_pack(1.0f, 1.0f)), d0, d1);
    f2_unpack(f2_mul(x, f2_pack(rcp_approx(d0), rcp_approx(d1))), y0, y1);
  } else {
    f2_unpack(x, y0, y1);
    if (e.act == 1) {
      y0 = fmaxf(y0, 0.0f);
      y1 = fmaxf(y1, 0.0f);
    }
  }
  return pack_bf16x2_rn(__float_as_uint(y0), __float_as_uint(y1));
}

// Bias of 8 consecutive columns starting at `col` (a multiple of 8) as 4 BF16 pairs; zero
// past N (N is a multiple of 8) or without a bias.
__device__ __forceinline__ uint4 epi_bias8(const EpiParams& e, int col, int N) {
  if (e.bias == nullptr || col >= N) return make_uint4(0u, 0u, 0u, 0u);
  return __ldg(reinterpret_cast<const uint4*>(e.bias + col));
}

}  // namespace dtcp

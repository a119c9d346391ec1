// gemm_nvfp4.cu -- NVFP4 block-scaled C = A * B^T on sm_103a tensor cores.
//
// A and B hold E2M1 codes (two per byte, K contiguous); the scales (one E4M3 per 16
// K-elements) arrive in the blocked layout of pack_scales.cu, in which one pipeline
// stage's scales for 128 rows are one contiguous 2 KB block. The block-scaled MMA
// (kind::mxf4nvf4, scale_vec::4X, K = 64 per instruction) reads the scales from TMEM;
// tcgen05.cp moves them there from shared memory.
//
// Persistent CTA pairs (cta_group::2), a 256 x 256 output tile per pair, 256 K-elements
// (128 bytes of codes per row, one 128-byte swizzle row) per pipeline stage. Every
// barrier wait, TMA issue, tcgen05.cp and tcgen05.mma costs its issuing thread tens to
// hundreds of cycles (a wait about 50-150, a copy about 25, an MMA about 75, a taken
// branch up to 200: the loops are straight-line code), and a stage keeps the tensor pipe
// busy only 512 cycles, so the per-stage work is spread over threads of different warps,
// each under that budget:
//   warp 0      TMA producer of A (both CTAs); arms the leader's full barrier
//   warp 1      TMA producer of B (both CTAs)
//   warp 2      TMA producer of SFA (this CTA's 128 rows) and SFB (all 256 rows, one 3-D box)
//               into the scale ring, whose slots the copiers' commits free
//   warp 3      MMA issuer (leader CTA) + TMEM allocator: one scale-ready wait per two
//               stages, 4 MMAs and a commit per stage
//   warps 4..11 epilogue: warp 4 + 4h + q reads TMEM lanes 32q.. of accumulator columns
//               128h..128h+127 into registers (four loads, one wait), releases TMEM, then
//               converts to BF16 and stores 32 x 16 tiles through a 1 KB staging buffer
//               (32-byte swizzled, conflict-free) with TMA (small, so that shared memory
//               holds a sixth stage)
//   warps 12..15 scale copiers (leader CTA): copier c copies the scales of MMA c of every
//               stage (SFA, SFB rows 0-127, SFB rows 128-255) and arrives on sf_ready as
//               soon as the copies are issued (copies and MMAs run in issue order)
// Shared memory: 6 A/B stages (32 KB each), a 4-slot scale ring (6 KB each) and 8 KB of C
// staging: the A/B ring covers the ~1300-cycle load latency of a stage with two stages
// to spare.
// Warpgroups 0 and 3 give up registers (setmaxnreg) to the epilogue warpgroups 1 and 2,
// which hold the whole 128 x 256 FP32 accumulator of a CTA in registers to free TMEM after
// a single load latency (the one TMEM slot is the MMAs' only accumulator).
// TMEM (512 columns): accumulator in columns 0..255 (one slot; the epilogue releases it as
// soon as it has read it); the 5-slot scale ring after it, 48 columns per slot (16 for SFA:
// 4 MMAs x 4 columns; 32 for SFB: 4 MMAs x 2 N-halves x 4 columns).
// A last wave at most half full runs as N-halves of its tiles (N = 128 MMAs).
//
// Design sources: "NVFP4 GEMM on Blackwell", Kernel 1 (warp roles, scales in TMEM via
// tcgen05.cp, 48-column scale buffers), Kernel 2 (CTA pairs: each CTA needs its own SFA
// half and all of SFB; leader-owned barriers; multicast commit), Kernel 3 (persistent
// grid, continuous stage counter, TMEM-empty handoff), Kernel 4 (epilogue reads all of
// TMEM before converting and releases it early).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "host_common.h"

namespace dtcp {

struct Nvfp4Params {
  int M, N, K;
  int num_m_blocks, num_n_blocks, num_tiles, k_iters;
  int split_tiles, num_items;  // trailing tiles cut into N-halves; work items = tiles + split_tiles
  int group_m;
  unsigned* status;
  unsigned long long wait_limit_ns;
  unsigned debug_flags;
  int zigzag;     // 1: the items of odd-numbered waves walk K downwards
  int wave;       // co-resident clusters
  int clc;        // 1: one cluster per item is launched; running clusters take the items of clusters they cancel
  EpiParams epi;  // fused epilogue (epi.fused == 0: plain BF16 rounding)
  ClockProbe probe;
};

template <int STAGES>
struct Nvfp4Layout {
  static constexpr int CG = 2;
  static constexpr int BLOCK_M = 128;              // output rows per CTA
  static constexpr int BLOCK_N = 256;              // output columns per tile
  static constexpr int BLOCK_K = 256;              // K elements per stage (128 bytes of codes)
  static constexpr int UMMA_K = 64;                // K per block-scaled MMA
  static constexpr int KSTEPS = BLOCK_K / UMMA_K;  // 4 MMAs per stage
  static constexpr int TILE_M = BLOCK_M * CG;
  static constexpr int B_ROWS = BLOCK_N / CG;      // B rows each CTA loads
  static constexpr int A_BYTES = BLOCK_M * BLOCK_K / 2;   // 16 KB
  static constexpr int B_BYTES = B_ROWS * BLOCK_K / 2;    // 16 KB
  static constexpr int SF_BLOCK = 512;                    // scales of 128 rows for one MMA
  static constexpr int SFA_BYTES = KSTEPS * SF_BLOCK;     // 2 KB: this CTA's 128 rows
  static constexpr int SFB_BYTES = 2 * KSTEPS * SF_BLOCK; // 4 KB: all 256 rows of the tile
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  // The scales have shallower rings than A and B: stage g uses A/B slot g % STAGES, scale
  // slot g % SF_SMEM_STAGES in shared memory (freed when its copies complete, well before
  // the stage's MMAs) and g % SF_STAGES in TMEM (5 slots fit beside the accumulator).
  static constexpr int SF_STAGES = STAGES < 5 ? STAGES : 5;
  static constexpr int SF_SMEM_STAGES = STAGES < 4 ? STAGES : 4;
  static constexpr int ACC_COLS = BLOCK_N;
  static constexpr int SF_COLS = KSTEPS * 4 + KSTEPS * 8;  // 16 + 32 TMEM columns per stage
  static constexpr int SF_TMEM_COL0 = ACC_COLS;
  static constexpr int TMEM_COLS = 512;
  // warp roles
  static constexpr int WARP_PROD_A = 0, WARP_PROD_B = 1, WARP_PROD_SF = 2, WARP_MMA = 3;
  // two epilogue warps per TMEM lane quadrant, one per 128-column half of the accumulator
  static constexpr int EPI_WARP0 = 4, EPI_WARPS = 8;
  static constexpr int COPY_WARP0 = 12, COPY_WARPS = KSTEPS;  // one copier per MMA of a stage
  static constexpr int NUM_THREADS = 32 * (COPY_WARP0 + COPY_WARPS);
  // registers per thread after setmaxnreg (the launch gives 65536 / 512 -> 128)
  static constexpr int REGS_LAUNCH = 128, REGS_LOW = 64, REGS_EPI = 184;

  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + SF_SMEM_STAGES * SFA_BYTES;
  static constexpr int OFF_EPI = OFF_SFB + SF_SMEM_STAGES * SFB_BYTES;
  // C staging per epilogue warp: 32 rows x 16 columns (one TMA store box)
  static constexpr int EPI_COLS = 16;
  static constexpr int EPI_BUF_BYTES = 32 * EPI_COLS * 2;
  static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * EPI_BUF_BYTES;
  // full[S], empty[S], sf_ready[S], sf_free[SF_SMEM_STAGES], tmem_full, tmem_empty, never, drain,
  // c_loaded[EPI_WARPS], clc_full[kClcSlots], clc_empty[kClcSlots]
  static constexpr int NUM_BARS = 3 * STAGES + SF_SMEM_STAGES + 4 + EPI_WARPS + 2 * kClcSlots;
  static constexpr int OFF_CLC = (OFF_BAR + NUM_BARS * 8 + 15) / 16 * 16;  // CLC responses, 16 bytes each
  // releases of a CLC response: producers B and SF and the epilogue warps of both CTAs, the
  // MMA issuer and the copiers (leader), and producer A of the second CTA (the leader's
  // issues the requests)
  static constexpr int CLC_CONSUMERS = CG * (2 + EPI_WARPS) + 1 + COPY_WARPS + 1;
  static constexpr int OFF_TMEM_SLOT = OFF_CLC + kClcSlots * 16;
  static constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
  static constexpr int SMEM_USED = OFF_ABORT + 4;
  static constexpr int SMEM_BYTES = SMEM_USED + 1024;

  static_assert(SMEM_BYTES <= 232448, "exceeds 227 KB of shared memory per CTA");
  static_assert(OFF_EPI % 1024 == 0 && EPI_BUF_BYTES % 256 == 0, "32-byte swizzled staging needs 256-byte alignment");
  static_assert(SF_TMEM_COL0 + SF_STAGES * SF_COLS <= TMEM_COLS, "scale ring does not fit in TMEM");
  static_assert(A_BYTES + B_BYTES == 32768, "A+B tile bytes per CTA per stage");
  static_assert(STAGE_BYTES == 38912, "38 KB stage of a CTA pair kernel");
  static_assert(NUM_THREADS == 512 && REGS_LAUNCH * NUM_THREADS <= 65536, "launch register budget");
  static_assert(128 * (2 * REGS_LOW + 2 * REGS_EPI) <= REGS_LAUNCH * NUM_THREADS,
                "setmaxnreg split exceeds the block's launch registers");
  static_assert(EPI_WARP0 % 4 == 0 && EPI_WARPS == 8 && COPY_WARP0 % 4 == 0, "roles must fill whole warpgroups");
};

// Barrier addresses and per-CTA context shared by the roles.
struct Nvfp4Ctx {
  uint32_t base;       // 1024-aligned shared-memory base (same offset in both CTAs)
  uint32_t warp, lane, rank;
  int cluster_idx, num_clusters;
  uint32_t tmem_base;
  uint32_t bar_full, bar_empty, bar_sfready, bar_sffree, bar_tfull, bar_tempty, bar_never, bar_drain, bar_cload;
  uint32_t bar_clc_empty;  // this CTA's clc_empty[0] (the leader's are the ones used)
  ClcRing ring;
  bool clc;
  WaitCtx wctx;
};

// First item of this cluster and the item after item `it` (static stride or CLC response
// `it`). `arm` / `release` as for clc_next; the roles here run under changed register
// limits, so the waits are inlined.
__device__ __forceinline__ int nvfp4_first_item(const Nvfp4Params& p, const Nvfp4Ctx& x) {
  return x.cluster_idx < p.num_items ? x.cluster_idx : -1;
}
__device__ __forceinline__ int nvfp4_next_item(const Nvfp4Params& p, const Nvfp4Ctx& x, int i, int it, bool arm,
                                               bool release, uint32_t code, bool& ok) {
  if (x.clc) return clc_next<true>(x.ring, it, 2, arm, release, x.wctx, code, ok);
  return i + x.num_clusters < p.num_items ? i + x.num_clusters : -1;
}

// ---------------------------------------------------------------- TMA producers (both CTAs)
// warp 0: A (and the leader arms the full barrier with the bytes of both CTAs); warp 1: B;
// warp 2: SFA and SFB. Each waits on its own CTA's empty barrier.
template <int STAGES>
__device__ __forceinline__ void producer_role(const Nvfp4Params& p, const CUtensorMap* tmap_a,
                                              const CUtensorMap* tmap_b, const CUtensorMap* tmap_b_half,
                                              const CUtensorMap* tmap_sfa, const CUtensorMap* tmap_sfb,
                                              const Nvfp4Ctx& x) {
  using L = Nvfp4Layout<STAGES>;
  if (x.lane != 0) return;
  const int ksteps = p.K / L::UMMA_K;  // 512-byte scale blocks per 128 rows
  uint32_t stage = 0, phase = 0;
  uint32_t sf_stage = 0, sf_phase = 0;  // the scale producer's slot in the scale ring
  bool ok = true;
  const bool is_a = x.warp == L::WARP_PROD_A;
  const bool issuer = x.clc && is_a && x.rank == 0;  // requests the CLC responses
  int it = 0;
  for (int i = nvfp4_first_item(p, x); i >= 0; ++it) {
    if (issuer && !clc_request<true, true>(x.ring, x.bar_clc_empty, it, x.wctx, status_code(kRoleProducer, 0x500 + it % kClcSlots))) {
      ok = false;
      break;
    }
    const WorkItem w = work_item(i, p.num_tiles, p.split_tiles);
    const TileCoord tc = tile_coord(w.tile, p.num_m_blocks, p.num_n_blocks, p.group_m);
    const bool half = w.half >= 0;
    // every other wave of items walks K downwards, so it starts on the K blocks the
    // previous wave read last (still in L2)
    const bool down = p.zigzag && (((x.clc ? i / p.wave : it) & 1) != 0);
    const int a_row = tc.m_blk * L::TILE_M + static_cast<int>(x.rank) * L::BLOCK_M;
    const int b_row = tc.n_blk * L::BLOCK_N + (half ? w.half * (L::BLOCK_N / 2) + static_cast<int>(x.rank) * (L::B_ROWS / 2)
                                                    : static_cast<int>(x.rank) * L::B_ROWS);
    const CUtensorMap* map_b = half ? tmap_b_half : tmap_b;
    // a half item loads half the B rows; the scales of the whole tile are loaded either way
    const uint32_t stage_bytes = L::STAGE_BYTES - (half ? L::B_BYTES / 2 : 0);
    const int sfa_block = (a_row / 128) * ksteps;
    // One straight-line loop per producer (the ring position and the K block advance by
    // selects): A and B issue one 2-D copy per stage, the scale producer a 2-D and a 3-D one.
    if (x.warp != L::WARP_PROD_SF) {
      static_assert(L::A_BYTES == L::B_BYTES, "A and B stages share one stride");
      const bool arm = is_a && x.rank == 0;  // one arrival with the bytes of both CTAs
      const uint32_t dst0 = x.base + (is_a ? L::OFF_A : L::OFF_B);
      const CUtensorMap* map = is_a ? tmap_a : map_b;
      const int row = is_a ? a_row : b_row;
#pragma unroll 2
      for (int kb = 0; kb < p.k_iters; ++kb) {
        // First pass over the ring: parity 1 of a fresh barrier counts as complete.
        if (!wait_phase_inline(x.bar_empty + 8 * stage, phase ^ 1u, x.wctx, status_code(kRoleProducer, (x.warp << 8) | stage))) {
          ok = false;
          break;
        }
        const uint32_t full = x.bar_full + 8 * stage;
        const int kblk = down ? p.k_iters - 1 - kb : kb;
        // the other loads may land before the arrival
        if (arm) mbar_arrive_expect_tx(full, 2 * stage_bytes);
        tma_load_2d_pair(dst0 + stage * L::A_BYTES, map, kblk * (L::BLOCK_K / 2), row, mapa_shared(full, 0));
        stage = stage + 1 == STAGES ? 0u : stage + 1;
        phase = stage == 0 ? phase ^ 1u : phase;
      }
    } else {
      // The scale slot is free once the copies of the stage that used it have completed
      // (the copiers commit to sf_free): earlier than that stage's MMAs.
#pragma unroll 2
      for (int kb = 0; kb < p.k_iters; ++kb) {
        if (!wait_phase_inline(x.bar_sffree + 8 * sf_stage, sf_phase ^ 1u, x.wctx, status_code(kRoleProducer, (x.warp << 8) | sf_stage))) {
          ok = false;
          break;
        }
        const uint32_t full_leader = mapa_shared(x.bar_full + 8 * stage, 0);
        const int kblk = down ? p.k_iters - 1 - kb : kb;
        const int ky = kblk * L::KSTEPS;  // scale blocks of this stage: 4 consecutive ones
        tma_load_2d_pair(x.base + L::OFF_SFA + sf_stage * L::SFA_BYTES, tmap_sfa, 0, sfa_block + ky, full_leader);
        // both 128-row blocks of the tile's SFB (row blocks 2n and 2n+1), steps ky .. ky+3
        tma_load_3d_pair(x.base + L::OFF_SFB + sf_stage * L::SFB_BYTES, tmap_sfb, 0, ky, tc.n_blk * 2, full_leader);
        stage = stage + 1 == STAGES ? 0u : stage + 1;
        sf_stage = sf_stage + 1 == L::SF_SMEM_STAGES ? 0u : sf_stage + 1;
        sf_phase = sf_stage == 0 ? sf_phase ^ 1u : sf_phase;
      }
    }
    if (!ok) break;
    // producer A re-arms this CTA's response slot for its next use
    i = nvfp4_next_item(p, x, i, it, is_a, !issuer, status_code(kRoleProducer, 0x600 + it % kClcSlots), ok);
  }
  if (!ok) settle_after_abort();
}

// ---------------------------------------------------------------- scale copiers (leader)
// Copier c moves, for every stage, the scale blocks of MMA c (SFA, SFB rows 0-127, SFB
// rows 128-255: 3 copies) from the stage's shared-memory scale slot to its TMEM scale slot,
// arrives on sf_ready, and commits the copies to sf_free (their completion frees the
// shared-memory slot for the scale producer). Before writing the TMEM slot it waits for the
// MMAs of the stage that used the slot last.
template <int STAGES>
__device__ __forceinline__ void copier_role(const Nvfp4Params& p, const Nvfp4Ctx& x) {
  using L = Nvfp4Layout<STAGES>;
  if (x.rank != 0 || x.lane != 0) return;
  const uint32_t c = x.warp - L::COPY_WARP0;
  const uint64_t sfa0 = umma_desc_advance(umma_desc_plain(x.base + L::OFF_SFA, 128), c * L::SF_BLOCK);
  const uint64_t sfb0 = umma_desc_advance(umma_desc_plain(x.base + L::OFF_SFB, 128), c * L::SF_BLOCK);
  const uint32_t col0 = x.tmem_base + L::SF_TMEM_COL0;
  uint32_t stage = 0, phase = 0;      // A/B ring: full and sf_ready barriers
  uint32_t sf_smem = 0;               // scale ring in shared memory
  uint32_t sf_stage = 0;              // scale ring in TMEM
  uint32_t e_stage = 0, e_phase = 0;  // A/B ring position of stage g - SF_STAGES
  // Stage g (counted over all of this cluster's items): false if a wait gave up.
  auto copy_stage = [&](long long g) -> bool {
    if (!wait_phase_inline(x.bar_full + 8 * stage, phase, x.wctx, status_code(kRoleScales, 0x300 + stage))) return false;
    if constexpr (L::SF_STAGES < STAGES) {
      // The TMEM slot's previous stage (g - SF_STAGES) must have completed its MMAs, which
      // read the scales there. (With equal rings the producers' wait implies it.)
      if (g >= L::SF_STAGES) {
        if (!wait_phase_inline(x.bar_empty + 8 * e_stage, e_phase, x.wctx, status_code(kRoleScales, 0x400 + e_stage)))
          return false;
        e_stage = e_stage + 1 == STAGES ? 0u : e_stage + 1;
        e_phase = e_stage == 0 ? e_phase ^ 1u : e_phase;
      }
    }
    const uint64_t sfa = umma_desc_advance(sfa0, sf_smem * L::SFA_BYTES);
    const uint64_t sfb = umma_desc_advance(sfb0, sf_smem * L::SFB_BYTES);
    const uint32_t col = col0 + sf_stage * L::SF_COLS;
    tc_fence_after_sync();
    tmem_cp_32x128b_warpx4<2>(col + 4 * c, sfa);
    tmem_cp_32x128b_warpx4<2>(col + 16 + 8 * c, sfb);
    tmem_cp_32x128b_warpx4<2>(col + 20 + 8 * c, umma_desc_advance(sfb, L::SFB_BYTES / 2));
    // tcgen05.cp and tcgen05.mma execute in issue order on the pair's tensor pipe: the MMAs
    // need only be issued after these copies, which the fence and the barrier (arrive here,
    // wait and fence::after_thread_sync in the MMA thread) establish. The MMA thread does
    // not wait for the copies to complete (a tcgen05.commit here would make it: -2.4%).
    tc_fence_before_sync();
    mbar_arrive_local(x.bar_sfready + 8 * stage);
    // the scale slot's shared memory (in both CTAs) is free once these copies complete
    mma_commit_pair_multicast(x.bar_sffree + 8 * sf_smem, 0x3);
    stage = stage + 1 == STAGES ? 0u : stage + 1;
    phase = stage == 0 ? phase ^ 1u : phase;
    sf_smem = sf_smem + 1 == L::SF_SMEM_STAGES ? 0u : sf_smem + 1;
    sf_stage = sf_stage + 1 == L::SF_STAGES ? 0u : sf_stage + 1;
    return true;
  };
  bool ok = true;
  if (!x.clc) {
    // static schedule: this cluster's stage count is known, one straight-line loop over all
    // of them (a per-item loop around it measured 2.7% slower)
    const int items = x.cluster_idx < p.num_items ? (p.num_items - x.cluster_idx + x.num_clusters - 1) / x.num_clusters : 0;
    const long long total = static_cast<long long>(items) * p.k_iters;
#pragma unroll 2
    for (long long g = 0; g < total; ++g) {
      if (!copy_stage(g)) {
        ok = false;
        break;
      }
    }
  } else {
    long long g = 0;
    int it = 0;
    for (int i = nvfp4_first_item(p, x); i >= 0; ++it) {
#pragma unroll 2
      for (int kb = 0; kb < p.k_iters; ++kb, ++g) {
        if (!copy_stage(g)) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
      i = nvfp4_next_item(p, x, i, it, false, true, status_code(kRoleScales, 0x600 + it % kClcSlots), ok);
    }
  }
  if (!ok) settle_after_abort();
}

// ---------------------------------------------------------------- MMA issuer (leader)
// The 4 MMAs of one stage and the commit that releases it when they have read it (shared
// memory and TMEM scales). Descriptors and scale columns follow from the ring position.
template <int STAGES>
__device__ __forceinline__ void mma_stage(const Nvfp4Ctx& x, uint64_t a_desc0, uint64_t b_desc0, uint32_t sf_col0,
                                          uint32_t idesc, uint32_t sfb_half_col, uint32_t stage, uint32_t sf_stage,
                                          bool first) {
  using L = Nvfp4Layout<STAGES>;
  const uint64_t a_desc = umma_desc_advance(a_desc0, stage * L::A_BYTES);
  const uint64_t b_desc = umma_desc_advance(b_desc0, stage * L::B_BYTES);
  const uint32_t sf_col = sf_col0 + sf_stage * L::SF_COLS;
#pragma unroll
  for (int j = 0; j < L::KSTEPS; ++j) {
    const uint32_t koff = j * (L::UMMA_K / 2);  // 32 bytes of packed codes per MMA
    mma_nvf4<2>(x.tmem_base, umma_desc_advance(a_desc, koff), umma_desc_advance(b_desc, koff), idesc, sf_col + 4 * j,
                sf_col + 16 + 8 * j + sfb_half_col, (first && j == 0) ? 0u : 1u);
  }
  mma_commit_pair_multicast(x.bar_empty + 8 * stage, 0x3);
}

// Two stages per scale-ready wait: each copier commits its stages in order, and a commit
// covers all earlier copies of its thread, so the scale-ready phase of the later stage
// implies the earlier one's; the copiers copied each stage only after its full barrier, so
// both stages' tiles are in shared memory too. The loop body is straight-line code (ring
// position by selects, no inner loop): each taken branch in this thread's loop cost it
// hundreds of cycles.
template <int STAGES>
__device__ __forceinline__ void mma_role(const Nvfp4Params& p, const Nvfp4Ctx& x) {
  using L = Nvfp4Layout<STAGES>;
  if (x.rank != 0 || x.lane != 0) return;
  constexpr uint32_t IDESC_FULL = idesc_nvf4(L::TILE_M, L::BLOCK_N);
  constexpr uint32_t IDESC_HALF = idesc_nvf4(L::TILE_M, L::BLOCK_N / 2);
  uint32_t stage = 0, phase = 0;  // A/B ring
  uint32_t sf_stage = 0;          // scale ring (TMEM slot)
  bool ok = true;
  if (p.debug_flags & 1u) ok = wait_phase_inline(x.bar_never, 0, x.wctx, status_code(kRoleMma, 0xFFFF));
  const uint64_t a_desc0 = umma_desc_sw128(x.base + L::OFF_A), b_desc0 = umma_desc_sw128(x.base + L::OFF_B);
  const uint32_t sf_col0 = x.tmem_base + L::SF_TMEM_COL0;
  int it = 0;
  for (int i = nvfp4_first_item(p, x); i >= 0 && ok; ++it) {
    const WorkItem w = work_item(i, p.num_tiles, p.split_tiles);
    const uint32_t idesc = w.half >= 0 ? IDESC_HALF : IDESC_FULL;
    const uint32_t sfb_half_col = w.half > 0 ? 4u : 0u;  // scale columns of the item's N-half
    if (!wait_phase_inline(x.bar_tempty, (static_cast<uint32_t>(it) & 1u) ^ 1u, x.wctx, status_code(kRoleMma, 0x100))) {
      ok = false;
      break;
    }
    tc_fence_after_sync();
    const int pairs = p.k_iters >> 1;
    int kb = 0;
#pragma unroll 2
    for (int q = 0; q < pairs; ++q, kb += 2) {
      const uint32_t s1 = stage + 1 == STAGES ? 0u : stage + 1;
      const uint32_t ph1 = s1 == 0 ? phase ^ 1u : phase;
      const uint32_t f1 = sf_stage + 1 == L::SF_STAGES ? 0u : sf_stage + 1;
      if (!wait_phase_inline(x.bar_sfready + 8 * s1, ph1, x.wctx, status_code(kRoleMma, 0x200 + s1))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      mma_stage<STAGES>(x, a_desc0, b_desc0, sf_col0, idesc, sfb_half_col, stage, sf_stage, kb == 0);
      mma_stage<STAGES>(x, a_desc0, b_desc0, sf_col0, idesc, sfb_half_col, s1, f1, false);
      stage = s1 + 1 == STAGES ? 0u : s1 + 1;
      phase = stage == 0 ? ph1 ^ 1u : ph1;
      sf_stage = f1 + 1 == L::SF_STAGES ? 0u : f1 + 1;
    }
    if (ok && kb < p.k_iters) {  // an odd number of stages: the last one alone
      if (!wait_phase_inline(x.bar_sfready + 8 * stage, phase, x.wctx, status_code(kRoleMma, 0x200 + stage))) {
        ok = false;
      } else {
        tc_fence_after_sync();
        mma_stage<STAGES>(x, a_desc0, b_desc0, sf_col0, idesc, sfb_half_col, stage, sf_stage, kb == 0);
        stage = stage + 1 == STAGES ? 0u : stage + 1;
        phase = stage == 0 ? phase ^ 1u : phase;
        sf_stage = sf_stage + 1 == L::SF_STAGES ? 0u : sf_stage + 1;
      }
    }
    if (!ok) break;
    mma_commit_pair_multicast(x.bar_tfull, 0x3);
    i = nvfp4_next_item(p, x, i, it, false, true, status_code(kRoleMma, 0x600 + it % kClcSlots), ok);
  }
  if (!ok) {
    mma_commit_pair_multicast(x.bar_drain, 0x1);
    const uint64_t t0 = globaltimer_ns();  // bounded: the issued MMAs finish or the limit passes
    while (!mbar_try_wait_suspend(x.bar_drain, 0, 20000u) && globaltimer_ns() - t0 < x.wctx.limit_ns) {
    }
    settle_after_abort();
  }
}

// ---------------------------------------------------------------- epilogue (warps 4..11)
// FUSED: the epilogue of the *_fused calls (its own kernel instantiation, so that the
// plain kernel's code stays as small as before).
template <int STAGES, bool FUSED>
__device__ __forceinline__ void epilogue_role(const Nvfp4Params& p, const CUtensorMap* tmap_c, const Nvfp4Ctx& x) {
  using L = Nvfp4Layout<STAGES>;
  const uint32_t lane = x.lane;
  const uint32_t q = x.warp & 3u;                  // this warp may access TMEM lanes 32q .. 32q+31
  const uint32_t epi = x.warp - L::EPI_WARP0;
  const int h = static_cast<int>(epi >> 2);        // accumulator columns 128h .. 128h+127
  const uint32_t buf = x.base + L::OFF_EPI + epi * L::EPI_BUF_BYTES;
  const uint32_t tempty_leader = mapa_shared(x.bar_tempty, 0);
  const uint32_t cload = x.bar_cload + 8 * epi;
  uint32_t cload_phase = 0;
  bool epi_ok = true;
  int it = 0;
  for (int i = nvfp4_first_item(p, x); i >= 0; ++it) {
    const WorkItem w = work_item(i, p.num_tiles, p.split_tiles);
    const TileCoord tc = tile_coord(w.tile, p.num_m_blocks, p.num_n_blocks, p.group_m);
    const int width = w.half >= 0 ? L::BLOCK_N / 2 : L::BLOCK_N;  // accumulator columns of the item
    int row0 = tc.m_blk * L::TILE_M + static_cast<int>(x.rank) * L::BLOCK_M + static_cast<int>(q) * 32;
    int col0 = tc.n_blk * L::BLOCK_N + (w.half > 0 ? L::BLOCK_N / 2 : 0) + h * 128;
    // The tile coordinates (integer divisions) are computed while the MMAs run, not after
    // the wait below, where they would delay the release of TMEM by ~450 cycles.
    asm volatile("" : "+r"(row0), "+r"(col0));
    if constexpr (FUSED) {
      // the prior C of this warp's part of the tile into L2 while the MMAs still run
      if (p.epi.beta != 0.0f && lane == 0 && row0 < p.M && h * 128 < width) {
#pragma unroll 1
        for (int e = 0; e < 128 / L::EPI_COLS; ++e)
          if (col0 + e * L::EPI_COLS < p.N) tma_prefetch_l2_2d(tmap_c, col0 + e * L::EPI_COLS, row0);
      }
    }
    if (__all_sync(0xffffffffu, wait_phase_inline(x.bar_tfull, static_cast<uint32_t>(it) & 1u, x.wctx,
                                                   status_code(kRoleEpilogue, 0))) == 0)
      break;
    tc_fence_after_sync();
    const uint32_t taddr = x.tmem_base + ((q * 32u) << 16) + static_cast<uint32_t>(h) * 128u;
    const bool live = row0 < p.M && h * 128 < width;
    uint32_t v[4][32];
    if (live) {
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(taddr + c * 32, v[c]);
      tmem_ld_wait();
    }
    // this warp's part of the accumulator is in registers: release TMEM, then convert and store
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader);  // orders tcgen05 work only
    if (live) {
      // 16 columns at a time: lane r writes its row's 32 bytes to the 32 x 16 staging tile,
      // one TMA store writes the tile (clipped at M and N)
#pragma unroll
      for (int e = 0; e < 128 / L::EPI_COLS; ++e) {
        const int col = col0 + e * L::EPI_COLS;
        if (col < p.N) {
          const uint32_t* s = &v[e >> 1][(e & 1) * 16];
          if (lane == 0) bulk_wait_group_read<0>();  // the store that last read `buf` is done
          __syncwarp();
          // Row `lane` of the 32 x 16 staging tile (32 bytes per row) with the 32-byte swizzle
          // of the C tensor map: 16-byte chunk j at j ^ (bit 2 of the row). The 8 lanes of a
          // store phase then cover all 32 banks (without it lanes r and r + 4 collide).
          const uint32_t row_addr = buf + lane * (L::EPI_COLS * 2);
          const uint32_t c0 = row_addr + (((lane >> 2) & 1u) << 4), c1 = c0 ^ 16u;
          uint32_t pk[8];
          if constexpr (!FUSED) {
#pragma unroll
            for (int k = 0; k < 8; ++k) pk[k] = pack_bf16x2_rn(s[2 * k], s[2 * k + 1]);
          } else {
            // prior C (beta != 0): the 32 x 16 tile by TMA into the staging buffer (zeros
            // past M and N), then row `lane` from it
            uint32_t old[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
            if (p.epi.beta != 0.0f) {
              if (lane == 0) {
                mbar_arrive_expect_tx(cload, L::EPI_BUF_BYTES);
                tma_load_2d(buf, tmap_c, col, row0, cload);
              }
              if (__all_sync(0xffffffffu, wait_phase_inline(cload, cload_phase, x.wctx,
                                                            status_code(kRoleEpilogue, 2))) == 0) {
                epi_ok = false;
                break;
              }
              cload_phase ^= 1u;
              ld_shared_v4(c0, old[0], old[1], old[2], old[3]);
              ld_shared_v4(c1, old[4], old[5], old[6], old[7]);
            }
            const uint4 b0 = epi_bias8(p.epi, col, p.N), b1 = epi_bias8(p.epi, col + 8, p.N);
            const uint32_t bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) pk[k] = epi_pair(s[2 * k], s[2 * k + 1], old[k], bb[k], p.epi);
            __syncwarp();  // every lane has read its row of the prior C before any lane overwrites it
          }
          st_shared_v4(c0, pk[0], pk[1], pk[2], pk[3]);
          st_shared_v4(c1, pk[4], pk[5], pk[6], pk[7]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(tmap_c, buf, col, row0);
            bulk_commit_group();
          }
        }
      }
    }
    if (!epi_ok) break;
    if (x.clc) {
      // every lane reads the response; one releases the slot
      const uint32_t s = static_cast<uint32_t>(it) % kClcSlots, ph = (static_cast<uint32_t>(it) / kClcSlots) & 1u;
      if (__all_sync(0xffffffffu, wait_phase_inline(x.ring.full + 8 * s, ph, x.wctx, status_code(kRoleEpilogue, 0x600 + s))) == 0)
        break;
      uint32_t cx;
      const bool got = clc_query(x.ring.resp + 16 * s, cx);
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(x.ring.empty_leader + 8 * s);
      i = got ? static_cast<int>(cx) / L::CG : -1;
    } else {
      i = i + x.num_clusters < p.num_items ? i + x.num_clusters : -1;
    }
  }
  if (lane == 0) bulk_wait_group<0>();
  __syncwarp();
}

// All roles meet here once their work is done; the MMA warp (which allocated TMEM) frees it.
template <int STAGES>
__device__ __forceinline__ void teardown(const Nvfp4Ctx& x) {
  tc_fence_before_sync();
  cluster_sync_all();
  if (x.warp == Nvfp4Layout<STAGES>::WARP_MMA) {
    tc_fence_after_sync();
    tmem_dealloc<2>(x.tmem_base, Nvfp4Layout<STAGES>::TMEM_COLS);
  }
}

// CLC: the instantiation with cluster launch control (p.clc == 1); the static one holds none
// of its code (the roles' tests of x.clc fold away).
template <int STAGES, bool FUSED, bool CLC>
__global__ void __launch_bounds__(Nvfp4Layout<STAGES>::NUM_THREADS, 1)
    nvfp4_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                      const __grid_constant__ CUtensorMap tmap_b_half, const __grid_constant__ CUtensorMap tmap_sfa,
                      const __grid_constant__ CUtensorMap tmap_sfb, const __grid_constant__ CUtensorMap tmap_c,
                      const Nvfp4Params p) {
  using L = Nvfp4Layout<STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  Nvfp4Ctx x;
  x.base = (raw + 1023u) & ~1023u;  // same offset in both CTAs of a pair
  uint8_t* smem = smem_raw + (x.base - raw);
  x.warp = threadIdx.x >> 5;
  x.lane = threadIdx.x & 31;
  x.rank = cluster_ctarank();
  x.cluster_idx = static_cast<int>(blockIdx.x) / L::CG;
  x.num_clusters = static_cast<int>(gridDim.x) / L::CG;
  x.bar_full = x.base + L::OFF_BAR;             // stage landed (leader's, bytes of both CTAs)
  x.bar_empty = x.bar_full + 8 * STAGES;        // stage consumed by the MMAs (both CTAs)
  x.bar_sfready = x.bar_empty + 8 * STAGES;     // stage's scales copied to TMEM (leader's)
  x.bar_sffree = x.bar_sfready + 8 * STAGES;    // scale slot's copies done (both CTAs, 4 commits)
  x.bar_tfull = x.bar_sffree + 8 * L::SF_SMEM_STAGES;  // accumulator ready
  x.bar_tempty = x.bar_tfull + 8;               // accumulator drained (leader's, 8 arrivals)
  x.bar_never = x.bar_tempty + 8;               // nobody arrives (timeout-path test)
  x.bar_drain = x.bar_never + 8;                // MMA drain after an abort
  x.bar_cload = x.bar_drain + 8;                // c_loaded[w]: epilogue warp w's prior-C tile landed
  const uint32_t bar_clc_full = x.bar_cload + 8 * L::EPI_WARPS;  // CLC response s landed here
  x.bar_clc_empty = bar_clc_full + 8 * kClcSlots;                // CLC response s released (leader's)
  x.ring = ClcRing{x.base + L::OFF_CLC, bar_clc_full, mapa_shared(x.bar_clc_empty, 0)};
  x.clc = CLC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEM_SLOT);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::OFF_ABORT);
  x.wctx = WaitCtx{abort_flag, p.status, p.wait_limit_ns};

  if (x.warp == 0 && x.lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(x.bar_full + 8 * s, 1);
      mbar_init(x.bar_empty + 8 * s, 1);
      mbar_init(x.bar_sfready + 8 * s, L::COPY_WARPS);
    }
    for (int s = 0; s < L::SF_SMEM_STAGES; ++s) mbar_init(x.bar_sffree + 8 * s, L::COPY_WARPS);
    mbar_init(x.bar_tfull, 1);
    mbar_init(x.bar_tempty, L::EPI_WARPS * L::CG);
    mbar_init(x.bar_never, 1);
    mbar_init(x.bar_drain, 1);
    for (int w = 0; w < L::EPI_WARPS; ++w) mbar_init(x.bar_cload + 8 * w, 1);
    for (int t = 0; t < kClcSlots; ++t) {
      mbar_init(bar_clc_full + 8 * t, 1);
      mbar_init(x.bar_clc_empty + 8 * t, L::CLC_CONSUMERS);
    }
    *abort_flag = 0u;
    fence_mbarrier_init_cluster();
    // every response slot armed for its first use (re-armed by producer A as it reads them)
    if (x.clc)
      for (int t = 0; t < kClcSlots; ++t) mbar_arrive_expect_tx(bar_clc_full + 8 * t, 16);
    prefetch_tensormap(&tmap_a);
    prefetch_tensormap(&tmap_b);
    prefetch_tensormap(&tmap_b_half);
    prefetch_tensormap(&tmap_sfa);
    prefetch_tensormap(&tmap_sfb);
    prefetch_tensormap(&tmap_c);
  }
  if (x.warp == L::WARP_MMA) {
    tmem_alloc<2>(smem_u32(tmem_slot), L::TMEM_COLS);
    tmem_relinquish<2>();
  }
  tc_fence_before_sync();
  cluster_sync_all();
  tc_fence_after_sync();
  x.tmem_base = *tmem_slot;
  // Set-up is done: the next kernel may start its own. Every global access below (TMA
  // loads and stores) comes after the previous kernel on the stream has completed.
  pdl_launch_dependents();
  pdl_wait();
  clock_probe_mark(p.probe, 0);

  // One branch per warpgroup, each with one register-limit change for all its warps: the
  // epilogue warpgroup takes the registers that warpgroups 0 and 2 give up. Each branch
  // runs to the end of the kernel (the code after a change of limit belongs to one limit).
  if (x.warp < L::EPI_WARP0) {
    regs_decrease<L::REGS_LOW>();
    if (x.warp <= L::WARP_PROD_SF) producer_role<STAGES>(p, &tmap_a, &tmap_b, &tmap_b_half, &tmap_sfa, &tmap_sfb, x);
    else mma_role<STAGES>(p, x);
    __syncwarp();
    teardown<STAGES>(x);
    clock_probe_mark(p.probe, 1);
  } else if (x.warp < L::COPY_WARP0) {
    regs_increase<L::REGS_EPI>();
    epilogue_role<STAGES, FUSED>(p, &tmap_c, x);
    teardown<STAGES>(x);
  } else {
    regs_decrease<L::REGS_LOW>();
    copier_role<STAGES>(p, x);
    __syncwarp();
    teardown<STAGES>(x);
  }
}

// ---------------------------------------------------------------------------- host side

namespace {

constexpr int kStages = 6;
using NL = Nvfp4Layout<kStages>;
constexpr auto kNvfp4Kernel = nvfp4_gemm_kernel<kStages, false, false>;
constexpr auto kNvfp4KernelFused = nvfp4_gemm_kernel<kStages, true, false>;
constexpr auto kNvfp4KernelClc = nvfp4_gemm_kernel<kStages, false, true>;
constexpr auto kNvfp4KernelFusedClc = nvfp4_gemm_kernel<kStages, true, true>;

int max_active_clusters(int device) {
  static std::mutex mu;
  static int cache[64] = {0};
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return 0;
  if (cache[device] > 0) return cache[device];
  for (auto k : {kNvfp4Kernel, kNvfp4KernelFused, kNvfp4KernelClc, kNvfp4KernelFusedClc})
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, NL::SMEM_BYTES) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(2 * 16, 1, 1);
  cfg.blockDim = dim3(NL::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = NL::SMEM_BYTES;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kNvfp4Kernel, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 0;
  }
  cache[device] = n;
  return n;
}

}  // namespace

int run_gemm_nvfp4_blocked(const void* A, const void* SFA, const void* B, const void* SFB, void* C, int M, int N,
                           int K, cudaStream_t stream, const RunOptions& opt, int a_rows) {
  int device = 0, err = 0;
  const DeviceInfo* info = current_device_info(&device, &err);
  if (info == nullptr) return err;
  if (opt.kernel != GEMM_KERNEL_DEFAULT) return GEMM_ERR_INVALID_ARG;

  CUtensorMap ta, tb, tbh, tsa, tsb, tc;
  const uint64_t kbytes = uint64_t(K) / 2;
  const uint64_t ksteps = uint64_t(K) / 64;
  int st = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, kbytes, std::max(M, a_rows), kbytes,
                          NL::BLOCK_K / 2, NL::BLOCK_M, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st == GEMM_OK)
    st = encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, kbytes, N, kbytes, NL::BLOCK_K / 2, NL::B_ROWS,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  if (st == GEMM_OK)  // B box of a half-width work item
    st = encode_tmap_2d(&tbh, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, kbytes, N, kbytes, NL::BLOCK_K / 2, NL::B_ROWS / 2,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  // blocked scales: rows of 512-byte blocks (128 words), one per (row block, 64-K step);
  // a box of 4 rows is one stage's scales for 128 rows
  if (st == GEMM_OK)
    st = encode_tmap_2d(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT32, SFA, 128, uint64_t(ceil_div(M, 128)) * ksteps, 512,
                        128, NL::KSTEPS, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st == GEMM_OK) {
    // SFB as [row block][64-K step][128 words]: one box holds a stage's 4 steps of both
    // row blocks of a 256-row tile, in the order the copiers read them
    const uint64_t dims[3] = {128, ksteps, uint64_t(ceil_div(N, 128))};
    const uint64_t strides[2] = {512, ksteps * 512};
    const uint32_t box[3] = {128, NL::KSTEPS, 2};
    st = encode_tmap_3d(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT32, SFB, dims, strides, box);
  }
  if (st == GEMM_OK)  // C stores: 32 rows x 16 columns of BF16 per box, 32-byte swizzle
    st = encode_tmap_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, C, N, M, uint64_t(N) * 2, NL::EPI_COLS, 32,
                        CU_TENSOR_MAP_SWIZZLE_32B);
  if (st != GEMM_OK) return st;

  Nvfp4Params p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.num_m_blocks = ceil_div(M, NL::TILE_M);
  p.num_n_blocks = ceil_div(N, NL::BLOCK_N);
  const long long tiles = static_cast<long long>(p.num_m_blocks) * p.num_n_blocks;
  if (tiles > 0x3FFFFFFFLL) return GEMM_ERR_UNSUPPORTED_SHAPE;
  p.num_tiles = static_cast<int>(tiles);
  p.k_iters = K / NL::BLOCK_K;
  p.status = device_status_word(device);
  p.wait_limit_ns = opt.wait_limit_ns;
  p.debug_flags = opt.debug_flags;
  p.zigzag = 1;
  p.epi.alpha = opt.epi.alpha;
  p.epi.beta = opt.epi.beta;
  p.epi.bias = static_cast<const uint16_t*>(opt.epi.bias);
  p.epi.act = opt.epi.act;
  p.epi.fused = opt.epi.fused() ? 1 : 0;
  p.probe = ClockProbe{opt.clock_probe, opt.clock_probe_ctas};
  if (p.status == nullptr) return GEMM_ERR_NO_DEVICE;

  const int max_clusters = max_active_clusters(device);
  if (max_clusters <= 0) return GEMM_ERR_LAUNCH;
  // Persistent grid: at most the co-resident clusters. The last partial wave is cut into
  // N-halves when they still fit in one wave.
  int wave = p.num_tiles;
  if (opt.persistent) {
    wave = max_clusters;
    if (opt.max_clusters > 0) wave = std::min(wave, opt.max_clusters);
  }
  p.split_tiles = (opt.persistent && opt.tail_split) ? tail_split_tiles(p.num_tiles, wave) : 0;
  p.num_items = p.num_tiles + p.split_tiles;
  // Cluster launch control: the whole grid of one cluster per item, taken dynamically
  p.clc = (opt.persistent && opt.max_clusters == 0 && use_clc(opt.clc, p.num_items, max_clusters, K, true)) ? 1 : 0;
  const int clusters = p.clc ? p.num_items : std::min(p.num_items, wave);
  p.wave = std::max(wave, 1);
  // bytes per row element: half a byte of code; plus one scale byte per 16 elements
  p.group_m = opt.group_m > 0 ? std::min(opt.group_m, p.num_m_blocks)
                              : choose_group_m(M, N, K, NL::TILE_M, NL::BLOCK_N, 0.5, 1.0 / 16.0, clusters,
                                               info->l2_bytes);

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * 2), 1, 1);
  cfg.blockDim = dim3(NL::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = NL::SMEM_BYTES;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = opt.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const auto kernel = p.clc ? (p.epi.fused ? kNvfp4KernelFusedClc : kNvfp4KernelClc)
                            : (p.epi.fused ? kNvfp4KernelFused : kNvfp4Kernel);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, ta, tb, tbh, tsa, tsb, tc, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  count_launch();
  return GEMM_OK;
}

}  // namespace dtcp

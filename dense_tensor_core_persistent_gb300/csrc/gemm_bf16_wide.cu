// gemm_bf16_wide.cu -- BF16 C = A * B^T with a 512 x 256 output tile per CTA pair: each
// CTA owns 256 rows of the tile as two 128-row M-waves, and the pair's cta_group::2 MMAs
// (M = 256, N = 256, K = 16) compute one wave of both CTAs at a time.
//
// Per 64-K stage each CTA loads A 256 x 64 (32 KB, one TMA box) and its half of B,
// 128 x 64 (16 KB): 48 KB per stage for 2 x 128 x 256 x 64 multiply-adds, where the
// 256 x 256 pair tile moves 64 KB per CTA for the same work (it re-reads A for every
// 256 columns and B for every 256 rows). So L2 -> shared-memory traffic falls by a
// quarter (M*N*K/85 bytes instead of M*N*K/64), and four stages (192 KB) hold three
// stages of MMA work in flight while one is refilled.
//
// The two waves' FP32 accumulators fill all 512 TMEM columns (wave w at columns 256w),
// so there is no second accumulator slot: the epilogue releases each wave's columns as
// soon as it has read them into registers, before storing, and the MMA issuer waits for
// wave 0's columns before the first MMA of a tile and for wave 1's columns before the
// first MMA of wave 1. Tile i's stores overlap tile i+1's MMAs.
//
// Warp roles (12 warps, three warpgroups): warp 0 TMA producer of A (arms the leader's full
// barrier with the bytes of both CTAs), warp 1 TMEM allocator and MMA issuer (leader CTA),
// warp 2 TMA producer of B; warps 4..11 epilogue, two per TMEM lane quadrant (warp % 4):
// warps 4..7 take columns 0..127 of each wave, warps 8..11 columns 128..255.
// Plain epilogue: a thread converts its 128 columns of a wave to 64 packed BF16 pairs as it
// reads them. Fused epilogue (FUSED): it keeps the 128 FP32 values (the epilogue's
// arithmetic comes before the one rounding), so the producer warpgroup gives up registers
// to the two epilogue warpgroups (setmaxnreg).
// A last wave of tiles at most half full runs as N-halves of its tiles (N = 128 MMAs).
//
// Design source: "Achieve cuBLAS Performance on NVIDIA GB300 for HGEMM", v7 (256 x 256
// per CTA as two 128-row M-waves whose accumulators fill TMEM side by side; a leader-owned
// load barrier armed with the cluster's bytes; the accumulator drained wave by wave
// through a two-buffer staging area and TMA stores); "NVFP4 GEMM on Blackwell", the
// epilogue section (bias, activation and alpha/beta scaling applied in the epilogue).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "host_common.h"

namespace dtcp {

struct WideParams {
  int M, N, K;
  int num_m_blocks, num_n_blocks, num_tiles, k_iters;
  int split_tiles, num_items;
  int group_m;
  unsigned* status;
  unsigned long long wait_limit_ns;
  unsigned debug_flags;
  int zigzag;
  EpiParams epi;  // fused epilogue (the FUSED instantiation)
  ClockProbe probe;
};

struct WideLayout {
  static constexpr int CG = 2;
  static constexpr int WAVES = 2;                    // 128-row M-waves per CTA
  static constexpr int WAVE_M = 128;                 // rows per wave per CTA (TMEM lanes)
  static constexpr int CTA_M = WAVE_M * WAVES;       // 256 rows of A per CTA
  static constexpr int TILE_M = CTA_M * CG;          // 512 rows per pair tile
  static constexpr int BLOCK_N = 256;                // MMA N, tile columns
  static constexpr int B_ROWS = BLOCK_N / CG;        // B rows each CTA loads
  static constexpr int BLOCK_K = 64;                 // one 128-byte swizzle row of BF16
  static constexpr int UMMA_K = 16;
  static constexpr int KSTEPS = BLOCK_K / UMMA_K;    // 4 MMAs per wave per stage
  static constexpr int STAGES = 4;
  static constexpr int A_WAVE_BYTES = WAVE_M * 128;  // 16 KB
  static constexpr int A_BYTES = CTA_M * 128;        // 32 KB
  static constexpr int B_BYTES = B_ROWS * 128;       // 16 KB
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int ACC_COLS = BLOCK_N;           // per wave
  static constexpr int TMEM_COLS = 512;
  static constexpr int WARP_PROD_A = 0, WARP_MMA = 1, WARP_PROD_B = 2;
  // two epilogue warps per TMEM lane quadrant, each for 128 of a wave's 256 columns
  static constexpr int EPI_WARP0 = 4, EPI_WARPS = 8;
  static constexpr int EPI_COLS = ACC_COLS / 2;      // columns per epilogue warp and wave
  static constexpr int EPI_BUFS = 2;
  static constexpr int STORE_COLS = 32;              // C store box: 32 rows x 32 BF16 columns
  static constexpr int EPI_BUF_BYTES = 32 * STORE_COLS * 2;  // 64-byte rows, 64-byte swizzle
  static constexpr int NUM_THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
  // registers per thread of the fused instantiation after setmaxnreg (the launch gives
  // 65536 / 384 -> 168): the producer warpgroup gives up registers to the epilogue ones
  static constexpr int REGS_LAUNCH = 168, REGS_LOW = 56, REGS_EPI = 216;

  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_EPI = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES;
  // full[S], empty[S], tmem_full, tmem_empty[WAVES], never, drain, c_loaded[EPI_WARPS]
  static constexpr int NUM_BARS = 2 * STAGES + 1 + WAVES + 2 + EPI_WARPS;
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
  static constexpr int SMEM_USED = OFF_ABORT + 4;
  static constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack to align the base to 1024 bytes

  static_assert(SMEM_BYTES <= 232448, "exceeds 227 KB of shared memory per CTA");
  static_assert(WAVES * ACC_COLS == TMEM_COLS, "the two waves' accumulators fill TMEM");
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0 && OFF_EPI % 1024 == 0, "1024-byte alignment");
  static_assert(CTA_M <= 256 && B_ROWS <= 256, "TMA box rows must not exceed 256");
  static_assert(EPI_WARP0 % 4 == 0 && EPI_WARPS == 8, "the epilogue fills whole warpgroups");
  static_assert(NUM_THREADS * REGS_LAUNCH <= 65536 && 128 * REGS_LOW + 256 * REGS_EPI <= NUM_THREADS * REGS_LAUNCH,
                "setmaxnreg split exceeds the block's launch registers");
};

// All lanes wait (each acquires what the barrier guards); the outcome is made uniform.
__device__ __forceinline__ bool wide_wait_warp(uint32_t bar, uint32_t parity, const WaitCtx& w, uint32_t code) {
  return __all_sync(0xffffffffu, wait_phase_inline(bar, parity, w, code)) != 0;
}

// ---------------------------------------------------------------- TMA producers (warps 0, 2)
__device__ __forceinline__ void wide_producer(const WideParams& p, const CUtensorMap* tmap_a, const CUtensorMap* tmap_b,
                                              const CUtensorMap* tmap_b_half, uint32_t base, uint32_t rank,
                                              bool load_a, int cluster_idx, int num_clusters, const WaitCtx& wctx) {
  using L = WideLayout;
  const uint32_t bar_full = base + L::OFF_BAR, bar_empty = bar_full + 8 * L::STAGES;
  uint32_t stage = 0, phase = 0;
  bool ok = true;
  int it = 0;
  for (int i = cluster_idx < p.num_items ? cluster_idx : -1; i >= 0; ++it) {
    const WorkItem w = work_item(i, p.num_tiles, p.split_tiles);
    const TileCoord tc = tile_coord(w.tile, p.num_m_blocks, p.num_n_blocks, p.group_m);
    const bool half = w.half >= 0;
    // every other item of a cluster walks K downwards: it starts on the K blocks the
    // previous wave of items read last (still in L2)
    const bool down = p.zigzag && ((it & 1) != 0);
    const int a_row = tc.m_blk * L::TILE_M + static_cast<int>(rank) * L::CTA_M;
    const int b_row = tc.n_blk * L::BLOCK_N + (half ? w.half * (L::BLOCK_N / 2) + static_cast<int>(rank) * (L::B_ROWS / 2)
                                                    : static_cast<int>(rank) * L::B_ROWS);
    const uint32_t stage_bytes = L::A_BYTES + (half ? L::B_BYTES / 2 : L::B_BYTES);
    const uint32_t dst0 = base + (load_a ? L::OFF_A : L::OFF_B);
    const uint32_t stride = load_a ? L::A_BYTES : L::B_BYTES;
    const CUtensorMap* map = load_a ? tmap_a : (half ? tmap_b_half : tmap_b);
    const int row = load_a ? a_row : b_row;
    const bool arm = load_a && rank == 0;  // one arrival with the bytes of both CTAs
#pragma unroll 2
    for (int kb = 0; kb < p.k_iters; ++kb) {
      // First pass over the ring: parity 1 of a fresh barrier counts as complete.
      if (!wait_phase_inline(bar_empty + 8 * stage, phase ^ 1u, wctx, status_code(kRoleProducer, stage))) {
        ok = false;
        break;
      }
      const uint32_t full = bar_full + 8 * stage;
      const int kblk = down ? p.k_iters - 1 - kb : kb;
      // the B loads may complete before the arrival; the phase cannot
      if (arm) mbar_arrive_expect_tx(full, 2u * stage_bytes);
      tma_load_2d_pair(dst0 + stage * stride, map, kblk * L::BLOCK_K, row, mapa_shared(full, 0));
      stage = stage + 1 == L::STAGES ? 0u : stage + 1;
      phase = stage == 0 ? phase ^ 1u : phase;
    }
    if (!ok) break;
    i = i + num_clusters < p.num_items ? i + num_clusters : -1;
  }
  if (!ok) settle_after_abort();
}

// ---------------------------------------------------------------- MMA issuer (leader, warp 1)
__device__ __forceinline__ void wide_mma(const WideParams& p, uint32_t base, uint32_t tmem_base, int cluster_idx,
                                         int num_clusters, const WaitCtx& wctx) {
  using L = WideLayout;
  const uint32_t bar_full = base + L::OFF_BAR, bar_empty = bar_full + 8 * L::STAGES;
  const uint32_t bar_tfull = bar_empty + 8 * L::STAGES, bar_tempty = bar_tfull + 8;
  const uint32_t bar_never = bar_tempty + 8 * L::WAVES, bar_drain = bar_never + 8;
  constexpr uint32_t IDESC_FULL = idesc_bf16(L::WAVE_M * L::CG, L::BLOCK_N);
  constexpr uint32_t IDESC_HALF = idesc_bf16(L::WAVE_M * L::CG, L::BLOCK_N / 2);
  uint32_t stage = 0, phase = 0;
  bool ok = true;
  if (p.debug_flags & 1u) ok = wait_phase_inline(bar_never, 0, wctx, status_code(kRoleMma, 0xFFFF));
  const uint64_t a_desc0 = umma_desc_sw128(base + L::OFF_A), b_desc0 = umma_desc_sw128(base + L::OFF_B);
  const uint32_t d0 = tmem_base, d1 = tmem_base + L::ACC_COLS;
  // The 4 MMAs of one wave for the stage at ring position `s` (accumulate unless `first`).
  auto wave_mmas = [&](uint32_t d, uint32_t s, uint32_t wave, uint32_t idesc, bool first) {
    const uint64_t a_desc = umma_desc_advance(a_desc0, s * L::A_BYTES + wave * L::A_WAVE_BYTES);
    const uint64_t b_desc = umma_desc_advance(b_desc0, s * L::B_BYTES);
#pragma unroll
    for (int kk = 0; kk < L::KSTEPS; ++kk)  // 32 bytes of K per MMA inside the 128-byte swizzle row
      mma_f16<2>(d, umma_desc_advance(a_desc, kk * 32), umma_desc_advance(b_desc, kk * 32), idesc,
                 (first && kk == 0) ? 0u : 1u);
  };
  int it = 0;
  for (int i = cluster_idx < p.num_items ? cluster_idx : -1; i >= 0 && ok; ++it) {
    const WorkItem w = work_item(i, p.num_tiles, p.split_tiles);
    const uint32_t idesc = w.half >= 0 ? IDESC_HALF : IDESC_FULL;
    const uint32_t acc_parity = (static_cast<uint32_t>(it) & 1u) ^ 1u;
    // first stage: wave 0 once its columns are free, wave 1 once its columns are free
    if (!wait_phase_inline(bar_tempty, acc_parity, wctx, status_code(kRoleMma, 0x100)) ||
        !wait_phase_inline(bar_full + 8 * stage, phase, wctx, status_code(kRoleMma, stage))) {
      ok = false;
      break;
    }
    tc_fence_after_sync();
    wave_mmas(d0, stage, 0, idesc, true);
    if (!wait_phase_inline(bar_tempty + 8, acc_parity, wctx, status_code(kRoleMma, 0x101))) {
      ok = false;
      break;
    }
    tc_fence_after_sync();
    wave_mmas(d1, stage, 1, idesc, true);
    mma_commit_pair_multicast(bar_empty + 8 * stage, 0x3);
    stage = stage + 1 == L::STAGES ? 0u : stage + 1;
    phase = stage == 0 ? phase ^ 1u : phase;
    // the other stages: straight-line (ring position by selects)
#pragma unroll 2
    for (int kb = 1; kb < p.k_iters; ++kb) {
      if (!wait_phase_inline(bar_full + 8 * stage, phase, wctx, status_code(kRoleMma, stage))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      wave_mmas(d0, stage, 0, idesc, false);
      wave_mmas(d1, stage, 1, idesc, false);
      // release the stage when these MMAs have read it; never wait here
      mma_commit_pair_multicast(bar_empty + 8 * stage, 0x3);
      stage = stage + 1 == L::STAGES ? 0u : stage + 1;
      phase = stage == 0 ? phase ^ 1u : phase;
    }
    if (!ok) break;
    mma_commit_pair_multicast(bar_tfull, 0x3);
    i = i + num_clusters < p.num_items ? i + num_clusters : -1;
  }
  if (!ok) {
    // let issued MMAs finish before TMEM is released (bounded: they finish or the limit passes)
    mma_commit_pair_multicast(bar_drain, 0x1);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_suspend(bar_drain, 0, 20000u) && globaltimer_ns() - t0 < wctx.limit_ns) {
    }
    settle_after_abort();
  }
}

// ---------------------------------------------------------------- epilogue (warps 4..11)
// One 32 x 32 chunk of this warp's rows: the packed BF16 pairs `pk` (columns 2j, 2j+1 in
// pk[j]) into the staging buffer (row `lane`, 16-byte chunk j at j ^ ((row / 2) % 4): the
// 64-byte swizzle of the C tensor map, which spreads the 8 lanes of a store phase over all
// 32 banks), then one TMA store.
__device__ __forceinline__ void wide_store_chunk(const CUtensorMap* tmap_c, uint32_t buf, uint32_t lane,
                                                 const uint32_t (&pk)[16], int col, int row0) {
  const uint32_t row_addr = buf + lane * 64u;
  const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ sw) << 4), pk[4 * j], pk[4 * j + 1], pk[4 * j + 2],
                 pk[4 * j + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmap_c, buf, col, row0);
    bulk_commit_group();
  }
}

template <bool FUSED>
__device__ __forceinline__ void wide_epilogue(const WideParams& p, const CUtensorMap* tmap_c, uint32_t base,
                                              uint32_t tmem_base, uint32_t warp, uint32_t lane, uint32_t rank,
                                              int cluster_idx, int num_clusters, const WaitCtx& wctx) {
  using L = WideLayout;
  const uint32_t bar_tfull = base + L::OFF_BAR + 16 * L::STAGES, bar_tempty = bar_tfull + 8;
  const uint32_t bar_cload = bar_tempty + 8 * L::WAVES + 16;
  const uint32_t q = warp & 3u;  // this warp may access TMEM lanes 32q .. 32q+31
  const uint32_t epi = warp - L::EPI_WARP0;
  const int h = static_cast<int>(epi >> 2);  // columns 128h .. 128h+127 of each wave
  const uint32_t stage_base = base + L::OFF_EPI + epi * L::EPI_BUFS * L::EPI_BUF_BYTES;
  const uint32_t tempty_leader = mapa_shared(bar_tempty, 0);
  const uint32_t cload = bar_cload + 8 * epi;
  uint32_t cload_phase = 0;
  bool epi_ok = true;
  uint32_t ebuf = 0;
  int it = 0;
  for (int i = cluster_idx < p.num_items ? cluster_idx : -1; i >= 0; ++it) {
    const WorkItem w = work_item(i, p.num_tiles, p.split_tiles);
    const TileCoord tc = tile_coord(w.tile, p.num_m_blocks, p.num_n_blocks, p.group_m);
    const int width = w.half >= 0 ? L::BLOCK_N / 2 : L::BLOCK_N;  // accumulator columns of the item
    const int row_cta = tc.m_blk * L::TILE_M + static_cast<int>(rank) * L::CTA_M + static_cast<int>(q) * 32;
    const int col0 = tc.n_blk * L::BLOCK_N + (w.half > 0 ? L::BLOCK_N / 2 : 0) + h * L::EPI_COLS;
    if constexpr (FUSED) {
      // the prior C of this warp's part of the tile into L2 while the MMAs still run
      if (p.epi.beta != 0.0f && lane == 0 && h * L::EPI_COLS < width) {
#pragma unroll 1
        for (int wv = 0; wv < L::WAVES; ++wv)
          if (row_cta + wv * L::WAVE_M < p.M)
            for (int c = 0; c < L::EPI_COLS / L::STORE_COLS; ++c)
              if (col0 + c * L::STORE_COLS < p.N)
                tma_prefetch_l2_2d(tmap_c, col0 + c * L::STORE_COLS, row_cta + wv * L::WAVE_M);
      }
    }
    if (!wide_wait_warp(bar_tfull, static_cast<uint32_t>(it) & 1u, wctx, status_code(kRoleEpilogue, 0))) break;
    tc_fence_after_sync();
#pragma unroll 1
    for (int wv = 0; wv < L::WAVES; ++wv) {
      const int row0 = row_cta + wv * L::WAVE_M;
      const bool live = row0 < p.M && h * L::EPI_COLS < width;
      const uint32_t taddr = tmem_base + ((q * 32u) << 16) + static_cast<uint32_t>(wv) * L::ACC_COLS +
                             static_cast<uint32_t>(h) * L::EPI_COLS;
      if constexpr (!FUSED) {
        // this lane's 128 columns of the wave as packed BF16 pairs: columns 2j, 2j+1 in pk[j]
        uint32_t pk[64];
        if (live) {
#pragma unroll
          for (int b = 0; b < 2; ++b) {  // two batches of 64 columns (two loads, one wait)
            uint32_t v[2][32];
#pragma unroll
            for (int c = 0; c < 2; ++c) tmem_ld_32x32b_x32(taddr + b * 64 + c * 32, v[c]);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int j = 0; j < 16; ++j) pk[b * 32 + c * 16 + j] = pack_bf16x2_rn(v[c][2 * j], v[c][2 * j + 1]);
          }
        }
        // this wave's columns are read: hand them back to the MMA issuer (leader's barrier)
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader + 8 * wv);  // orders tcgen05 work only
        if (live) {
#pragma unroll
          for (int c = 0; c < L::EPI_COLS / L::STORE_COLS; ++c) {
            const int col = col0 + c * L::STORE_COLS;
            if (col < p.N) {
              const uint32_t buf = stage_base + ebuf * L::EPI_BUF_BYTES;
              if (lane == 0) bulk_wait_group_read<1>();  // the store that last read `buf` is done
              __syncwarp();
              uint32_t chunk[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) chunk[j] = pk[c * 16 + j];
              wide_store_chunk(tmap_c, buf, lane, chunk, col, row0);
              ebuf ^= 1u;
            }
          }
        }
      } else {
        // the 128 FP32 values of this lane's row: the epilogue's arithmetic comes before
        // the one rounding, so they stay in registers after TMEM is released
        uint32_t v[4][32];
        if (live) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(taddr + c * 32, v[c]);
          tmem_ld_wait();
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader + 8 * wv);  // orders tcgen05 work only
        if (live) {
#pragma unroll
          for (int c = 0; c < L::EPI_COLS / L::STORE_COLS; ++c) {
            const int col = col0 + c * L::STORE_COLS;
            if (col < p.N) {
              const uint32_t buf = stage_base + ebuf * L::EPI_BUF_BYTES;
              if (lane == 0) bulk_wait_group_read<1>();  // the store that last read `buf` is done
              __syncwarp();
              const uint32_t row_addr = buf + lane * 64u;
              const uint32_t sw = (lane >> 1) & 3u;
              // prior C (beta != 0): the 32 x 32 chunk by TMA into the staging buffer (zeros
              // past M and N, same swizzle as the store), then row `lane` from it
              uint32_t old[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) old[j] = 0u;
              if (p.epi.beta != 0.0f) {
                if (lane == 0) {
                  mbar_arrive_expect_tx(cload, L::EPI_BUF_BYTES);
                  tma_load_2d(buf, tmap_c, col, row0, cload);
                }
                if (!wide_wait_warp(cload, cload_phase, wctx, status_code(kRoleEpilogue, 2))) {
                  epi_ok = false;
                  break;
                }
                cload_phase ^= 1u;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  ld_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ sw) << 4), old[4 * j], old[4 * j + 1],
                               old[4 * j + 2], old[4 * j + 3]);
              }
              uint32_t pk[16];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint4 bb = epi_bias8(p.epi, col + 8 * j, p.N);
                const uint32_t b4[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
                for (int t = 0; t < 4; ++t)
                  pk[4 * j + t] = epi_pair(v[c][8 * j + 2 * t], v[c][8 * j + 2 * t + 1], old[4 * j + t], b4[t], p.epi);
              }
              __syncwarp();  // every lane has read its row of the prior C before any lane overwrites it
              wide_store_chunk(tmap_c, buf, lane, pk, col, row0);
              ebuf ^= 1u;
            }
          }
        }
        if (!epi_ok) break;
      }
    }
    if (!epi_ok) break;
    i = i + num_clusters < p.num_items ? i + num_clusters : -1;
  }
  if (lane == 0) bulk_wait_group<0>();
  __syncwarp();
}

// All roles meet here once their work is done; the MMA warp (which allocated TMEM) frees it.
__device__ __forceinline__ void wide_teardown(uint32_t warp, uint32_t tmem_base) {
  tc_fence_before_sync();
  cluster_sync_all();
  if (warp == WideLayout::WARP_MMA) {
    tc_fence_after_sync();
    tmem_dealloc<2>(tmem_base, WideLayout::TMEM_COLS);
  }
}

template <bool FUSED>
__global__ void __launch_bounds__(WideLayout::NUM_THREADS, 1)
    bf16_wide_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                          const __grid_constant__ CUtensorMap tmap_b_half, const __grid_constant__ CUtensorMap tmap_c,
                          const WideParams p) {
  using L = WideLayout;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // same offset in both CTAs of a pair
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster_idx = static_cast<int>(blockIdx.x) / L::CG;
  const int num_clusters = static_cast<int>(gridDim.x) / L::CG;

  const uint32_t bar_full = base + L::OFF_BAR;         // full[s]: stage s loaded (leader's copy used)
  const uint32_t bar_empty = bar_full + 8 * L::STAGES;  // empty[s]: stage s consumed by the MMAs
  const uint32_t bar_tfull = bar_empty + 8 * L::STAGES; // tmem_full: both waves' accumulators ready
  const uint32_t bar_tempty = bar_tfull + 8;            // tmem_empty[w]: wave w's columns read (leader's)
  const uint32_t bar_never = bar_tempty + 8 * L::WAVES; // nobody arrives (timeout-path test)
  const uint32_t bar_drain = bar_never + 8;             // MMA drain after an abort
  const uint32_t bar_cload = bar_drain + 8;             // c_loaded[w]: epilogue warp w's prior-C chunk landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEM_SLOT);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::OFF_ABORT);
  const WaitCtx wctx{abort_flag, p.status, p.wait_limit_ns};

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_tfull, 1);
    for (int w = 0; w < L::WAVES; ++w) mbar_init(bar_tempty + 8 * w, L::EPI_WARPS * L::CG);
    mbar_init(bar_never, 1);
    mbar_init(bar_drain, 1);
    for (int w = 0; w < L::EPI_WARPS; ++w) mbar_init(bar_cload + 8 * w, 1);
    *abort_flag = 0u;
    fence_mbarrier_init_cluster();
    prefetch_tensormap(&tmap_a);
    prefetch_tensormap(&tmap_b);
    prefetch_tensormap(&tmap_b_half);
    prefetch_tensormap(&tmap_c);
  }
  if (warp == L::WARP_MMA) {
    tmem_alloc<2>(smem_u32(tmem_slot), L::TMEM_COLS);
    tmem_relinquish<2>();
  }
  tc_fence_before_sync();
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // Set-up is done: the next kernel may start its own. Every global access below (TMA
  // loads and stores) comes after the previous kernel on the stream has completed.
  pdl_launch_dependents();
  pdl_wait();
  clock_probe_mark(p.probe, 0);

  // One branch per role group, each running to the end of the kernel (with FUSED, the
  // code after a change of register limit belongs to that limit).
  if (warp < L::EPI_WARP0) {
    if constexpr (FUSED) regs_decrease<L::REGS_LOW>();
    if (lane == 0) {
      if (warp == L::WARP_PROD_A || warp == L::WARP_PROD_B)
        wide_producer(p, &tmap_a, &tmap_b, &tmap_b_half, base, rank, warp == L::WARP_PROD_A, cluster_idx,
                      num_clusters, wctx);
      else if (warp == L::WARP_MMA && rank == 0)
        wide_mma(p, base, tmem_base, cluster_idx, num_clusters, wctx);
    }
    __syncwarp();
    wide_teardown(warp, tmem_base);
    clock_probe_mark(p.probe, 1);
  } else {
    if constexpr (FUSED) regs_increase<L::REGS_EPI>();
    wide_epilogue<FUSED>(p, &tmap_c, base, tmem_base, warp, lane, rank, cluster_idx, num_clusters, wctx);
    wide_teardown(warp, tmem_base);
  }
}

// ---------------------------------------------------------------------------- host side

namespace {

int wide_max_active_clusters(int device) {
  static std::mutex mu;
  static int cache[64] = {0};
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return 0;
  if (cache[device] > 0) return cache[device];
  for (auto k : {bf16_wide_gemm_kernel<false>, bf16_wide_gemm_kernel<true>})
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, WideLayout::SMEM_BYTES) != cudaSuccess)
      return 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(2 * 16, 1, 1);
  cfg.blockDim = dim3(WideLayout::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = WideLayout::SMEM_BYTES;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, bf16_wide_gemm_kernel<false>, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 0;
  }
  cache[device] = n;
  return n;
}

}  // namespace

int run_gemm_bf16_wide(const void* A, const void* B, void* C, int M, int N, int K, cudaStream_t stream,
                       const RunOptions& opt) {
  using L = WideLayout;
  int device = 0, err = 0;
  const DeviceInfo* info = current_device_info(&device, &err);
  if (info == nullptr) return err;
  if (opt.clc == 1) return GEMM_ERR_INVALID_ARG;  // static schedule only
  CUtensorMap ta, tb, tbh, tc;
  int st = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, K, M, uint64_t(K) * 2, L::BLOCK_K, L::CTA_M,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  if (st == GEMM_OK)
    st = encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, K, N, uint64_t(K) * 2, L::BLOCK_K, L::B_ROWS,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  if (st == GEMM_OK)  // B box of a half-width work item
    st = encode_tmap_2d(&tbh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, K, N, uint64_t(K) * 2, L::BLOCK_K, L::B_ROWS / 2,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  if (st == GEMM_OK)  // C stores (and prior-C loads): 32 rows x 32 columns, 64-byte swizzle
    st = encode_tmap_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, C, N, M, uint64_t(N) * 2, L::STORE_COLS, 32,
                        CU_TENSOR_MAP_SWIZZLE_64B);
  if (st != GEMM_OK) return st;

  WideParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.num_m_blocks = ceil_div(M, L::TILE_M);
  p.num_n_blocks = ceil_div(N, L::BLOCK_N);
  const long long tiles = static_cast<long long>(p.num_m_blocks) * p.num_n_blocks;
  if (tiles > 0x3FFFFFFFLL) return GEMM_ERR_UNSUPPORTED_SHAPE;
  p.num_tiles = static_cast<int>(tiles);
  p.k_iters = ceil_div(K, L::BLOCK_K);
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

  const int max_clusters = wide_max_active_clusters(device);
  if (max_clusters <= 0) return GEMM_ERR_LAUNCH;
  int wave = p.num_tiles;
  if (opt.persistent) {
    wave = max_clusters;
    if (opt.max_clusters > 0) wave = std::min(wave, opt.max_clusters);
  }
  p.split_tiles = (opt.persistent && opt.tail_split) ? tail_split_tiles(p.num_tiles, wave) : 0;
  p.num_items = p.num_tiles + p.split_tiles;
  const int clusters = std::min(p.num_items, wave);
  p.group_m = opt.group_m > 0 ? std::min(opt.group_m, p.num_m_blocks)
                              : choose_group_m(M, N, K, L::TILE_M, L::BLOCK_N, 2.0, 0.0, clusters, info->l2_bytes);

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * L::CG), 1, 1);
  cfg.blockDim = dim3(L::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = L::SMEM_BYTES;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = L::CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = opt.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const auto kernel = p.epi.fused ? bf16_wide_gemm_kernel<true> : bf16_wide_gemm_kernel<false>;
  if (cudaLaunchKernelEx(&cfg, kernel, ta, tb, tbh, tc, p) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  count_launch();
  return GEMM_OK;
}

}  // namespace dtcp

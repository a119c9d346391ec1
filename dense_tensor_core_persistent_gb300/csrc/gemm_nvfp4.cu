// gemm_nvfp4.cu -- NVFP4 block-scaled C = A * B^T on sm_103a tensor cores.
//
// A and B hold E2M1 codes (two per byte), SFA / SFB one E4M3 scale per 16 K-elements
// (row-major [rows][K/16]). The block-scaled MMA (kind::mxf4nvf4, scale_vec::4X, K = 64
// per instruction) applies the scales; it reads them from TMEM, so every stage's scales
// travel global -> shared (TMA) -> shared, rearranged (scale-factor warp) -> TMEM
// (tcgen05.cp, issued in order with the MMAs that use them).
//
// Persistent CTA pairs (cta_group::2), a 256 x 256 output tile per pair, 256 K-elements
// (128 bytes of codes per row, one 128-byte swizzle row) per pipeline stage:
//   warp 0      TMA producer for A / B: 16 KB of A and 16 KB of B per CTA per stage
//   warp 1      MMA issuer (leader CTA) + TMEM allocator: 12 tcgen05.cp + 4 MMAs per stage
//   warps 2..5  epilogue: all TMEM loads first, early release, then BF16 TMA stores
//   warp 6      scale-factor producer: TMA of the row-major scale tiles into a landing
//               buffer, rearrangement into the tcgen05.cp source layout
// TMEM (512 columns): accumulator in columns 0..255; the scale ring after it, 48 columns
// per stage (16 for SFA: 4 MMAs x 4 columns; 32 for SFB: 4 MMAs x 2 N-halves x 4).
//
// Design sources: "NVFP4 GEMM on Blackwell", Kernel 1 (warp roles, scales in TMEM via
// tcgen05.cp in the MMA warp, 48-column scale buffers), Kernel 2 (CTA pairs, each CTA
// needs its own SFA half and all of SFB, scales waited for before the tiles), Kernel 3
// (persistent grid, continuous stage counter, TMEM-empty handoff), Kernel 4 (epilogue
// reads all of TMEM before converting, releases it early).
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
  int group_m;
  unsigned* status;
  unsigned long long wait_limit_ns;
  unsigned debug_flags;
};

// BLOCKED = false: scales arrive row-major ([rows][K/16]) and a scale warp rearranges them.
// BLOCKED = true:  scales arrive already in the tcgen05.cp source layout (see
//                  pack_scales.cu), so a stage's scales for 128 rows are one contiguous
//                  2 KB block that the producer loads with the tiles.
template <int STAGES, bool BLOCKED>
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
  static constexpr int SF_PER_ROW = BLOCK_K / 16;         // 16 scale bytes per row per stage
  static constexpr int SFA_BYTES = BLOCK_M * SF_PER_ROW;  // 2 KB (this CTA's rows)
  static constexpr int SFB_BYTES = BLOCK_N * SF_PER_ROW;  // 4 KB (all 256 rows of the tile)
  static constexpr int SF_BLOCK = 512;                    // one tcgen05.cp source: 128 rows x 4 scales
  static constexpr int ACC_COLS = BLOCK_N;
  static constexpr int SF_COLS = KSTEPS * 4 + KSTEPS * 8;  // 16 + 32 TMEM columns per stage
  static constexpr int SF_TMEM_COL0 = ACC_COLS;
  static constexpr int TMEM_COLS = 512;
  static constexpr int EPI_WARPS = 4;
  static constexpr int EPI_BUFS = 2;
  static constexpr int EPI_BUF_BYTES = 32 * 64 * 2;
  static constexpr int SF_WARP = 2 + EPI_WARPS;            // warp 6 (row-major scales only)
  // Scale-copy warps (leader CTA): one thread issues a tcgen05.cp only every ~56 cycles,
  // so the 12 copies of a stage are spread over 2 warps (copier c handles MMAs 2c, 2c+1:
  // SFA and both SFB halves) and the MMA thread issues only MMAs.
  static constexpr int COPY_WARPS = 2;
  static constexpr int COPY_WARP0 = SF_WARP + (BLOCKED ? 0 : 1);
  static constexpr int NUM_THREADS = 32 * (COPY_WARP0 + COPY_WARPS);
  static constexpr int LAND_STAGES = BLOCKED ? 0 : STAGES;

  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;       // rearranged, tcgen05.cp source
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
  static constexpr int OFF_SFA_IN = OFF_SFB + STAGES * SFB_BYTES; // TMA landing, row-major
  static constexpr int OFF_SFB_IN = OFF_SFA_IN + LAND_STAGES * SFA_BYTES;
  static constexpr int OFF_EPI = OFF_SFB_IN + LAND_STAGES * SFB_BYTES;
  static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES;
  // full[S], empty[S], sf_landed[S], sf_full[S], sf_ready[S], tmem_full, tmem_empty, never, drain
  static constexpr int NUM_BARS = 5 * STAGES + 4;
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
  static constexpr int SMEM_USED = OFF_ABORT + 4;
  static constexpr int SMEM_BYTES = SMEM_USED + 1024;

  static_assert(SMEM_BYTES <= 232448, "exceeds 227 KB of shared memory per CTA");
  static_assert(SF_TMEM_COL0 + STAGES * SF_COLS <= TMEM_COLS, "scale ring does not fit in TMEM");
  static_assert(SFA_BYTES == 4 * SF_BLOCK && SFB_BYTES == 8 * SF_BLOCK, "scale block arithmetic");
  static_assert(A_BYTES + B_BYTES == 32768, "A+B tile bytes per CTA per stage");
  static_assert(A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES == 38912, "38 KB stage of a CTA pair kernel");
};

// Rearrange one 128-row block of row-major scales (16 bytes per row: 4 MMAs x 4 scales)
// into the four 512-byte tcgen05.cp sources, one per MMA. In source j, the 16-byte line
// r holds the 4 scales of MMA j for rows r, r+32, r+64, r+96 (the .32x128b.warpx4 copy
// puts line r into TMEM lane r of every 32-lane quadrant, and quadrant q's MMA rows read
// the q-th 32-bit column).
__device__ __forceinline__ void rearrange_scale_block(uint32_t src_rows, uint32_t dst_blocks, uint32_t lane) {
  uint32_t w[4][4];
#pragma unroll
  for (int qd = 0; qd < 4; ++qd)
    ld_shared_v4(src_rows + (lane + 32u * qd) * 16u, w[qd][0], w[qd][1], w[qd][2], w[qd][3]);
#pragma unroll
  for (int j = 0; j < 4; ++j) st_shared_v4(dst_blocks + j * 512u + lane * 16u, w[0][j], w[1][j], w[2][j], w[3][j]);
}

template <int STAGES, bool BLOCKED>
__global__ void __launch_bounds__(Nvfp4Layout<STAGES, BLOCKED>::NUM_THREADS, 1)
    nvfp4_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                      const __grid_constant__ CUtensorMap tmap_sfa, const __grid_constant__ CUtensorMap tmap_sfb,
                      const __grid_constant__ CUtensorMap tmap_c, const Nvfp4Params p) {
  using L = Nvfp4Layout<STAGES, BLOCKED>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster_idx = static_cast<int>(blockIdx.x) / L::CG;
  const int num_clusters = static_cast<int>(gridDim.x) / L::CG;

  const uint32_t bar_full = base + L::OFF_BAR;          // A/B of a stage landed (leader's, pair bytes)
  const uint32_t bar_empty = bar_full + 8 * STAGES;     // stage consumed by the MMAs (both CTAs)
  const uint32_t bar_sfland = bar_empty + 8 * STAGES;   // scale TMA landed (each CTA's own)
  const uint32_t bar_sffull = bar_sfland + 8 * STAGES;  // rearranged scales ready (leader's, 2 arrivals)
  const uint32_t bar_sfready = bar_sffull + 8 * STAGES; // scales copied to TMEM (leader's, 3 commits)
  const uint32_t bar_tfull = bar_sfready + 8 * STAGES;  // accumulator ready
  const uint32_t bar_tempty = bar_tfull + 8;            // accumulator drained (leader's, 8 arrivals)
  const uint32_t bar_never = bar_tempty + 8;
  const uint32_t bar_drain = bar_never + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEM_SLOT);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::OFF_ABORT);
  const WaitCtx wctx{abort_flag, p.status, p.wait_limit_ns};

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
      mbar_init(bar_sfland + 8 * s, 1);
      mbar_init(bar_sffull + 8 * s, L::CG);
      mbar_init(bar_sfready + 8 * s, L::COPY_WARPS);
    }
    mbar_init(bar_tfull, 1);
    mbar_init(bar_tempty, L::EPI_WARPS * L::CG);
    mbar_init(bar_never, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0u;
    fence_mbarrier_init_cluster();
    prefetch_tensormap(&tmap_a);
    prefetch_tensormap(&tmap_b);
    prefetch_tensormap(&tmap_sfa);
    prefetch_tensormap(&tmap_sfb);
    prefetch_tensormap(&tmap_c);
  }
  if (warp == 1) {
    tmem_alloc<2>(smem_u32(tmem_slot), L::TMEM_COLS);
    tmem_relinquish<2>();
  }
  tc_fence_before_sync();
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ A/B TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int t = cluster_idx; t < p.num_tiles && ok; t += num_clusters) {
        const TileCoord tc = tile_coord(t, p.num_m_blocks, p.num_n_blocks, p.group_m);
        const int a_row = tc.m_blk * L::TILE_M + static_cast<int>(rank) * L::BLOCK_M;
        const int b_row = tc.n_blk * L::BLOCK_N + static_cast<int>(rank) * L::B_ROWS;
        for (int kb = 0; kb < p.k_iters; ++kb) {
          if (!wait_phase(bar_empty + 8 * stage, phase ^ 1u, wctx, status_code(kRoleProducer, stage))) {
            ok = false;
            break;
          }
          const uint32_t full = bar_full + 8 * stage;
          constexpr uint32_t kStageBytes = L::A_BYTES + L::B_BYTES + (BLOCKED ? L::SFA_BYTES + L::SFB_BYTES : 0);
          if (rank == 0) mbar_arrive_expect_tx(full, 2 * kStageBytes);
          const uint32_t full_leader = mapa_shared(full, 0);
          tma_load_2d_pair(base + L::OFF_A + stage * L::A_BYTES, &tmap_a, kb * (L::BLOCK_K / 2), a_row, full_leader);
          tma_load_2d_pair(base + L::OFF_B + stage * L::B_BYTES, &tmap_b, kb * (L::BLOCK_K / 2), b_row, full_leader);
          if constexpr (BLOCKED) {
            // 512-byte blocks indexed (row block, 64-K step); one stage = 4 consecutive blocks
            const int ksteps = p.K / L::UMMA_K;
            const int y = kb * L::KSTEPS;
            tma_load_2d_pair(base + L::OFF_SFA + stage * L::SFA_BYTES, &tmap_sfa, 0, (a_row / 128) * ksteps + y,
                             full_leader);
#pragma unroll
            for (int h = 0; h < 2; ++h)
              tma_load_2d_pair(base + L::OFF_SFB + stage * L::SFB_BYTES + h * 2048, &tmap_sfb, 0,
                               (tc.n_blk * 2 + h) * ksteps + y, full_leader);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) settle_after_abort();
    }
    __syncwarp();
  } else if (!BLOCKED && warp == L::SF_WARP) {
    // ------------------------------------------------------------ scale-factor producer
    // Landing buffer s is refilled (TMA for stage g+STAGES) as soon as this warp has
    // rearranged stage g out of it; only the rearranged buffer, which tcgen05.cp reads,
    // has to wait for the MMAs of stage g-STAGES (empty barrier). The loads therefore
    // run STAGES ahead and never wait behind MMA completion.
    const int k_iters = p.k_iters;
    const int my_tiles = (p.num_tiles - cluster_idx + num_clusters - 1) / num_clusters;
    const long long total = static_cast<long long>(my_tiles > 0 ? my_tiles : 0) * k_iters;
    const uint32_t sffull_leader = mapa_shared(bar_sffull, 0);
    auto issue = [&](long long gi) {
      if (lane == 0) {
        const uint32_t s = static_cast<uint32_t>(gi % STAGES);
        const int tile = cluster_idx + static_cast<int>(gi / k_iters) * num_clusters;
        const int kb = static_cast<int>(gi % k_iters);
        const TileCoord tc = tile_coord(tile, p.num_m_blocks, p.num_n_blocks, p.group_m);
        const int a_row = tc.m_blk * L::TILE_M + static_cast<int>(rank) * L::BLOCK_M;
        const int b_row = tc.n_blk * L::BLOCK_N;
        const uint32_t land = bar_sfland + 8 * s;
        mbar_arrive_expect_tx(land, L::SFA_BYTES + L::SFB_BYTES);
        tma_load_2d(base + L::OFF_SFA_IN + s * L::SFA_BYTES, &tmap_sfa, kb * L::SF_PER_ROW, a_row, land);
        tma_load_2d(base + L::OFF_SFB_IN + s * L::SFB_BYTES, &tmap_sfb, kb * L::SF_PER_ROW, b_row, land);
      }
      __syncwarp();
    };
    for (long long gi = 0; gi < total && gi < STAGES; ++gi) issue(gi);
    bool ok = true;
    for (long long g = 0; g < total; ++g) {
      const uint32_t s = static_cast<uint32_t>(g % STAGES);
      const uint32_t ph = static_cast<uint32_t>((g / STAGES) & 1);
      if (!wait_phase_warp(bar_sfland + 8 * s, ph, wctx, status_code(kRoleScales, 0x100 + s)) ||
          !wait_phase_warp(bar_empty + 8 * s, ph ^ 1u, wctx, status_code(kRoleScales, s))) {
        ok = false;
        break;
      }
      rearrange_scale_block(base + L::OFF_SFA_IN + s * L::SFA_BYTES, base + L::OFF_SFA + s * L::SFA_BYTES, lane);
#pragma unroll
      for (int h = 0; h < 2; ++h)
        rearrange_scale_block(base + L::OFF_SFB_IN + s * L::SFB_BYTES + h * 2048,
                              base + L::OFF_SFB + s * L::SFB_BYTES + h * 2048, lane);
      fence_proxy_async_smem();  // generic-proxy writes -> tcgen05.cp reads
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(sffull_leader + 8 * s);
      if (g + STAGES < total) issue(g + STAGES);  // landing buffer s is free again
    }
    if (!ok) settle_after_abort();
    __syncwarp();
  } else if (warp >= L::COPY_WARP0) {
    // ------------------------------------------------------------ scale copiers (leader)
    // Copier c moves, for every stage, the scale blocks of MMAs 2c and 2c+1 (SFA, SFB rows
    // 0-127, SFB rows 128-255: 6 copies) from shared memory to the stage's TMEM scale
    // slot, then commits to sf_ready. Waiting for
    // the stage's data (full / sf_full) also guarantees the MMAs STAGES stages earlier,
    // which read the same TMEM slot, have completed (the data could not be reloaded before).
    const int c = static_cast<int>(warp) - L::COPY_WARP0;
    if (rank == 0 && lane == 0) {
      const int my_tiles = (p.num_tiles - cluster_idx + num_clusters - 1) / num_clusters;
      const long long total = static_cast<long long>(my_tiles > 0 ? my_tiles : 0) * p.k_iters;
      const uint32_t data_bar = BLOCKED ? bar_full : bar_sffull;
      const uint64_t sfa0 = umma_desc_plain(base + L::OFF_SFA, 128), sfb0 = umma_desc_plain(base + L::OFF_SFB, 128);
      uint64_t sfa = sfa0, sfb = sfb0;
      uint32_t col = tmem_base + L::SF_TMEM_COL0;
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (long long g = 0; g < total; ++g) {
        if (!wait_phase(data_bar + 8 * stage, phase, wctx, status_code(kRoleScales, 0x300 + stage))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll
        for (int jj = 0; jj < L::KSTEPS / L::COPY_WARPS; ++jj) {
          const uint32_t j = c * (L::KSTEPS / L::COPY_WARPS) + jj;
          tmem_cp_32x128b_warpx4<2>(col + 4 * j, umma_desc_advance(sfa, j * L::SF_BLOCK));
          tmem_cp_32x128b_warpx4<2>(col + 16 + 8 * j, umma_desc_advance(sfb, j * L::SF_BLOCK));
          tmem_cp_32x128b_warpx4<2>(col + 20 + 8 * j, umma_desc_advance(sfb, 2048 + j * L::SF_BLOCK));
        }
        mma_commit_pair_multicast(bar_sfready + 8 * stage, 0x1);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
          sfa = sfa0;
          sfb = sfb0;
          col = tmem_base + L::SF_TMEM_COL0;
        } else {
          sfa = umma_desc_advance(sfa, L::SFA_BYTES);
          sfb = umma_desc_advance(sfb, L::SFB_BYTES);
          col += L::SF_COLS;
        }
      }
      if (!ok) settle_after_abort();
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (rank == 0 && lane == 0) {
      constexpr uint32_t IDESC = idesc_nvf4(L::TILE_M, L::BLOCK_N);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      if (p.debug_flags & 1u) ok = wait_phase(bar_never, 0, wctx, status_code(kRoleMma, 0xFFFF));
      int it = 0;
      // Per-stage operand descriptors and scale columns, advanced with the ring position
      // instead of being rebuilt from addresses for every instruction.
      const uint64_t a_desc0 = umma_desc_sw128(base + L::OFF_A), b_desc0 = umma_desc_sw128(base + L::OFF_B);
      const uint32_t sf_col0 = tmem_base + L::SF_TMEM_COL0;
      uint64_t a_desc = a_desc0, b_desc = b_desc0;
      uint32_t sf_col = sf_col0;
      for (int t = cluster_idx; t < p.num_tiles && ok; t += num_clusters, ++it) {
        if (!wait_phase(bar_tempty, (static_cast<uint32_t>(it) & 1u) ^ 1u, wctx, status_code(kRoleMma, 0x100))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        for (int kb = 0; kb < p.k_iters; ++kb) {
          // the stage's scales are in TMEM (copy warps) and its tiles in shared memory
          if (!wait_phase(bar_sfready + 8 * stage, phase, wctx, status_code(kRoleMma, 0x200 + stage)) ||
              !wait_phase(bar_full + 8 * stage, phase, wctx, status_code(kRoleMma, stage))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll
          for (int j = 0; j < L::KSTEPS; ++j) {
            const uint32_t koff = j * (L::UMMA_K / 2);  // 32 bytes of packed codes per MMA
            mma_nvf4<2>(tmem_base, umma_desc_advance(a_desc, koff), umma_desc_advance(b_desc, koff), IDESC,
                        sf_col + 4 * j, sf_col + 16 + 8 * j, (kb | j) != 0 ? 1u : 0u);
          }
          mma_commit_pair_multicast(bar_empty + 8 * stage, 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
            a_desc = a_desc0;
            b_desc = b_desc0;
            sf_col = sf_col0;
          } else {
            a_desc = umma_desc_advance(a_desc, L::A_BYTES);
            b_desc = umma_desc_advance(b_desc, L::B_BYTES);
            sf_col += L::SF_COLS;
          }
        }
        if (!ok) break;
        mma_commit_pair_multicast(bar_tfull, 0x3);
      }
      if (!ok) {
        mma_commit_pair_multicast(bar_drain, 0x1);
        wait_phase_slow(bar_drain, 0, wctx, status_code(kRoleMma, 0xFFFE), false);
        settle_after_abort();
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const uint32_t q = warp & 3u;
    const uint32_t epi = warp - 2u;
    const uint32_t stage_base = base + L::OFF_EPI + epi * L::EPI_BUFS * L::EPI_BUF_BYTES;
    const uint32_t tempty_leader = mapa_shared(bar_tempty, 0);
    uint32_t ebuf = 0;
    int it = 0;
    for (int t = cluster_idx; t < p.num_tiles; t += num_clusters, ++it) {
      const TileCoord tc = tile_coord(t, p.num_m_blocks, p.num_n_blocks, p.group_m);
      if (!wait_phase_warp(bar_tfull, static_cast<uint32_t>(it) & 1u, wctx, status_code(kRoleEpilogue, 0))) break;
      tc_fence_after_sync();
      const int row0 = tc.m_blk * L::TILE_M + static_cast<int>(rank) * L::BLOCK_M + static_cast<int>(q) * 32;
      const int col0 = tc.n_blk * L::BLOCK_N;
      const uint32_t taddr = tmem_base + ((q * 32u) << 16);
      const bool rows_live = row0 < p.M;
      uint32_t pk[4][32];
      if (rows_live) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t lo[32], hi[32];
          tmem_ld_32x32b_x32(taddr + c * 64, lo);
          tmem_ld_32x32b_x32(taddr + c * 64 + 32, hi);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            pk[c][i] = pack_bf16x2_rn(lo[2 * i], lo[2 * i + 1]);
            pk[c][16 + i] = pack_bf16x2_rn(hi[2 * i], hi[2 * i + 1]);
          }
        }
      }
      // whole accumulator is in registers: release TMEM before converting/storing
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader);
      if (rows_live) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int col = col0 + c * 64;
          if (col < p.N) {
            const uint32_t buf = stage_base + ebuf * L::EPI_BUF_BYTES;
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
            const uint32_t row_addr = buf + lane * 128u;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4), pk[c][4 * j],
                           pk[c][4 * j + 1], pk[c][4 * j + 2], pk[c][4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmap_c, buf, col, row0);
              bulk_commit_group();
            }
            ebuf ^= 1u;
          }
        }
      }
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  tc_fence_before_sync();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc<2>(tmem_base, L::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------- host side

namespace {

template <int STAGES, bool BLOCKED>
struct Nvfp4Variant {
  using L = Nvfp4Layout<STAGES, BLOCKED>;
  static constexpr auto kernel = nvfp4_gemm_kernel<STAGES, BLOCKED>;

  static int max_active_clusters(int device) {
    static std::mutex mu;
    static int cache[64] = {0};
    std::lock_guard<std::mutex> lock(mu);
    if (device < 0 || device >= 64) return 0;
    if (cache[device] > 0) return cache[device];
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_BYTES) != cudaSuccess)
      return 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(2 * 16, 1, 1);
    cfg.blockDim = dim3(L::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM_BYTES;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return 0;
    }
    cache[device] = n;
    return n;
  }

  static int run(const void* A, const void* SFA, const void* B, const void* SFB, void* C, int M, int N, int K,
                 cudaStream_t stream, const RunOptions& opt, int device, const DeviceInfo& info) {
    CUtensorMap ta, tb, tsa, tsb, tc;
    const uint64_t kbytes = uint64_t(K) / 2, kscales = uint64_t(K) / 16;
    int st = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, kbytes, M, kbytes, L::BLOCK_K / 2, L::BLOCK_M,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == GEMM_OK)
      st = encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, kbytes, N, kbytes, L::BLOCK_K / 2, L::B_ROWS,
                          CU_TENSOR_MAP_SWIZZLE_128B);
    if (BLOCKED) {
      // blocked scales: rows of 512-byte blocks (128 words), one block per (row block, 64-K step)
      const uint64_t ksteps = uint64_t(K) / 64;
      if (st == GEMM_OK)
        st = encode_tmap_2d(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT32, SFA, 128, uint64_t(ceil_div(M, 128)) * ksteps,
                            512, 128, L::KSTEPS, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (st == GEMM_OK)
        st = encode_tmap_2d(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT32, SFB, 128, uint64_t(ceil_div(N, 128)) * ksteps,
                            512, 128, L::KSTEPS, CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {
      if (st == GEMM_OK)
        st = encode_tmap_2d(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT8, SFA, kscales, M, kscales, L::SF_PER_ROW, L::BLOCK_M,
                            CU_TENSOR_MAP_SWIZZLE_NONE);
      if (st == GEMM_OK)
        st = encode_tmap_2d(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT8, SFB, kscales, N, kscales, L::SF_PER_ROW, L::BLOCK_N,
                            CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (st == GEMM_OK)
      st = encode_tmap_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, C, N, M, uint64_t(N) * 2, 64, 32,
                          CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != GEMM_OK) return st;

    Nvfp4Params p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.num_m_blocks = ceil_div(M, L::TILE_M);
    p.num_n_blocks = ceil_div(N, L::BLOCK_N);
    const long long tiles = static_cast<long long>(p.num_m_blocks) * p.num_n_blocks;
    if (tiles > 0x7FFFFFFFLL) return GEMM_ERR_UNSUPPORTED_SHAPE;
    p.num_tiles = static_cast<int>(tiles);
    p.k_iters = K / L::BLOCK_K;
    p.status = device_status_word(device);
    p.wait_limit_ns = opt.wait_limit_ns;
    p.debug_flags = opt.debug_flags;
    if (p.status == nullptr) return GEMM_ERR_NO_DEVICE;

    const int max_clusters = max_active_clusters(device);
    if (max_clusters <= 0) return GEMM_ERR_LAUNCH;
    int clusters = p.num_tiles;
    if (opt.persistent) {
      clusters = std::min(clusters, max_clusters);
      if (opt.max_clusters > 0) clusters = std::min(clusters, opt.max_clusters);
    }
    // bytes per row element: half a byte of code; plus one scale byte per 16 elements
    p.group_m = opt.group_m > 0 ? std::min(opt.group_m, p.num_m_blocks)
                                : choose_group_m(M, N, K, L::TILE_M, L::BLOCK_N, 0.5, 1.0 / 16.0, clusters,
                                                 info.l2_bytes);

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * 2), 1, 1);
    cfg.blockDim = dim3(L::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM_BYTES;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, ta, tb, tsa, tsb, tc, p);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_LAUNCH;
    }
    count_launch();
    return GEMM_OK;
  }
};

using Nvfp4RowMajorScales = Nvfp4Variant<4, false>;
using Nvfp4BlockedScales = Nvfp4Variant<5, true>;

}  // namespace

int run_gemm_nvfp4(const void* A, const void* SFA, const void* B, const void* SFB, void* C, int M, int N, int K,
                   cudaStream_t stream, const RunOptions& opt, bool blocked_scales) {
  int device = 0, err = 0;
  const DeviceInfo* info = current_device_info(&device, &err);
  if (info == nullptr) return err;
  if (opt.kernel != GEMM_KERNEL_DEFAULT) return GEMM_ERR_INVALID_ARG;
  if (blocked_scales) return Nvfp4BlockedScales::run(A, SFA, B, SFB, C, M, N, K, stream, opt, device, *info);
  return Nvfp4RowMajorScales::run(A, SFA, B, SFB, C, M, N, K, stream, opt, device, *info);
}

}  // namespace dtcp

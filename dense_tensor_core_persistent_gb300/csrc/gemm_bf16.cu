// gemm_bf16.cu -- BF16 C = A * B^T on sm_103a tensor cores (tcgen05), FP32 accumulation:
// the 256 x 256 pair tile (and its 1-CTA, swapped few-row and split-K variants) and the
// host dispatch between it and the 512 x 256 pair tile of gemm_bf16_wide.cu.
//
// One persistent, warp-specialised kernel template:
//   warp 0      TMA producer of A: fills an S-stage shared-memory ring with A K-slices and
//               arms the stage's full barrier
//   warp 6      TMA producer of B (its own thread, so a stage's loads go out sooner)
//   warp 1      MMA issuer (one thread of the pair's leader CTA) + TMEM allocator
//   warps 2..5  epilogue: TMEM -> registers -> BF16 -> swizzled smem -> TMA store
// CG = 1: one CTA computes a 128 x 256 tile (MMA M = 128).
// CG = 2: a CTA pair computes a 256 x 256 tile with cta_group::2 MMAs (M = 256): each
//         CTA holds 128 rows of A and 128 rows (N-half) of B per stage, the leader's
//         barrier counts the bytes of both CTAs, and MMA completion is multicast to both.
// The TMEM accumulator is double buffered (2 x 256 columns): the epilogue of tile i
// drains one slot while the MMAs of tile i+1 fill the other.
// A stage holds ATOMS columns of 64 K (one 128-byte swizzle row each). The default pair
// kernel uses 3 stages of 128 K, 8 MMAs per barrier wait: the issuing thread spends about
// 230 cycles per stage on the wait, fence and commit besides ~60 per MMA, so with 4 MMAs
// (512 pipe cycles) per stage it can barely keep the tensor pipe fed.
//
// Fused epilogue (gemm_bf16_fused): act(alpha * acc + beta * C + bias) before the rounding;
// the prior C of a chunk comes by TMA into the staging buffer (epi_pair, common.cuh).
//
// Few rows (M <= 128, N >= 256): the host runs the SWAP instantiations on (B, A), so the
// kernel computes C^T = B A^T with tile N 64 or 128 and its epilogue writes each 64 x 32
// chunk transposed into C. When such a GEMM has at most a third as many tiles as clusters,
// its K is split: each split writes FP32 partial sums to a workspace and
// splitk_reduce_transposed adds them.
//
// Design sources: "Achieve cuBLAS Performance on NVIDIA GB300 for HGEMM" (v1 swizzled
// TMA + descriptor, v3 warp specialisation with full/empty barriers, v4 2-CTA cluster
// MMA with multicast commit, v5 persistent kernel with a two-slot TMEM pipeline, v6
// TMA-store epilogue with two staging buffers and grouped tile order); "Optimized B200
// Matrix Multiplication" (section 4: the MMA issuer never waits for its own MMAs; it
// commits to the stage's empty barrier and the producer waits only when it wraps);
// "NVFP4 GEMM on Blackwell" (Kernel 2: leader-owned barriers, cluster-scope waits;
// Kernel 3: continuous stage/phase counter across tiles and the TMEM-empty handoff).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "host_common.h"

namespace dtcp {

struct Bf16Params {
  int M, N, K;
  int num_m_blocks, num_n_blocks, num_tiles, k_iters;
  int split_tiles, num_items;  // trailing tiles cut into N-halves; work items = tiles + split_tiles
  int group_m;
  unsigned* status;
  unsigned long long wait_limit_ns;
  unsigned debug_flags;
  int zigzag;  // 1: the items of odd-numbered waves walk K downwards
  int wave;    // co-resident clusters
  EpiParams epi;  // fused epilogue (epi.fused == 0: plain BF16 rounding)
  // split K (swapped variants): work item i is split i % splits of tile i / splits, over
  // stages [split * k_per_split, ...); each writes its FP32 partial tile to ws (row r of the
  // tile at ws + (split * M + r) * ldw); a second kernel sums and rounds them
  int splits, k_per_split, ldw;
  float* ws;
  int clc;  // 1: one cluster per item is launched; running clusters take the items of clusters they cancel
  ClockProbe probe;
};

struct Bf16Item {
  int tile, half;  // as WorkItem
  int split, k0, kn;  // K split, its first stage and its number of stages
};

__device__ __forceinline__ Bf16Item bf16_item(const Bf16Params& p, int i, bool split_k) {
  Bf16Item r;
  if (split_k && p.splits > 1) {
    r.tile = i / p.splits;
    r.split = i - r.tile * p.splits;
    r.half = -1;
    r.k0 = r.split * p.k_per_split;
    r.kn = min(p.k_per_split, p.k_iters - r.k0);
  } else {
    const WorkItem w = work_item(i, p.num_tiles, p.split_tiles);
    r.tile = w.tile;
    r.half = w.half;
    r.split = 0;
    r.k0 = 0;
    r.kn = p.k_iters;
  }
  return r;
}

// BN: output columns per tile (the MMA N). SWAP: the kernel computes C^T = B A^T for a
// GEMM with few rows (its A and B arguments are the caller's B and A) and writes each
// accumulator chunk transposed into the caller's C.
template <int CG, int STAGES, int ATOMS, int BN = 256, bool SWAP = false>
struct Bf16Layout {
  static constexpr int BLOCK_M = 128;              // output rows per CTA = TMEM lanes
  static constexpr int BLOCK_N = BN;               // output columns per tile = MMA N
  static constexpr int ATOM_K = 64;                // BF16 elements of one 128-byte swizzle row
  static constexpr int BLOCK_K = ATOM_K * ATOMS;   // K elements per stage
  static constexpr int UMMA_K = 16;                // K per tcgen05.mma kind::f16
  static constexpr int KSTEPS = BLOCK_K / UMMA_K;  // MMAs per stage
  static constexpr int TILE_M = BLOCK_M * CG;      // output rows per tile (per CTA pair for CG = 2)
  static constexpr int B_ROWS = BLOCK_N / CG;      // rows of B each CTA loads per stage
  static constexpr int A_ATOM_BYTES = BLOCK_M * 128;  // one swizzle-row column of the A tile
  static constexpr int B_ATOM_BYTES = B_ROWS * 128;
  static constexpr int A_BYTES = A_ATOM_BYTES * ATOMS;
  static constexpr int B_BYTES = B_ATOM_BYTES * ATOMS;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int ACC_COLS = BLOCK_N;         // FP32 accumulator columns per TMEM slot
  static constexpr int TMEM_COLS = 2 * ACC_COLS;   // two slots
  static constexpr int EPI_WARPS = 4;
  static constexpr int EPI_BUFS = 2;
  static constexpr int EPI_BUF_BYTES = 32 * 64 * 2;  // 32 rows x 64 BF16 columns (one swizzle row each)
  static constexpr int WARP_PROD_B = 2 + EPI_WARPS;  // warp 6
  static constexpr int NUM_THREADS = 32 * (3 + EPI_WARPS);

  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_EPI = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES;
  // barriers: full[S], empty[S], tmem_full[2], tmem_empty[2], never, drain, c_loaded[EPI_WARPS],
  // clc_full[kClcSlots], clc_empty[kClcSlots], partner (two pairs per cluster: the second
  // pair's partial sums are in the workspace)
  static constexpr int NUM_BARS = 2 * STAGES + 4 + 2 + EPI_WARPS + 2 * kClcSlots + 1;
  static constexpr int OFF_CLC = (OFF_BAR + NUM_BARS * 8 + 15) / 16 * 16;  // CLC responses, 16 bytes each
  // releases of a CLC response: producer B of each CTA, the MMA issuer, the epilogue warps
  // of each CTA, and for a pair producer A of the second CTA (the leader's issues them)
  static constexpr int CLC_CONSUMERS = CG * (1 + EPI_WARPS) + 1 + (CG - 1);
  static constexpr int OFF_TMEM_SLOT = OFF_CLC + kClcSlots * 16;
  static constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
  static constexpr int SMEM_USED = OFF_ABORT + 4;
  static constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack to align the base to 1024 bytes

  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "stage tiles must keep 1024-byte alignment");
  static_assert(SMEM_BYTES <= 232448, "exceeds 227 KB of shared memory per CTA");
  static_assert(TMEM_COLS <= 512, "exceeds the 512 TMEM columns of an SM");
  static_assert(B_ROWS <= 256, "TMA box rows must not exceed 256");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "tile N: 64, 128, 192 or 256 (whole 64-column epilogue chunks)");
};

// CLC: the instantiation with cluster launch control (p.clc == 1); the static one holds none
// of its code. PAIRS = 2 or 4 (swapped, that many K splits): a cluster of PAIRS CTA pairs
// computes one tile, pair s the s-th part of K; pairs 1 .. PAIRS-1 write their FP32 partial
// sums to the workspace and signal the first pair's epilogue, which adds them (in split
// order) before rounding. The pairs of a cluster run at the same time, so no second kernel
// is needed.
template <int CG, int STAGES, int ATOMS, int BN, bool SWAP, bool CLC, int PAIRS>
__global__ void __launch_bounds__(Bf16Layout<CG, STAGES, ATOMS, BN, SWAP>::NUM_THREADS, 1)
    bf16_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                     const __grid_constant__ CUtensorMap tmap_b_half, const __grid_constant__ CUtensorMap tmap_c,
                     const Bf16Params p) {
  using L = Bf16Layout<CG, STAGES, ATOMS, BN, SWAP>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // same offset in both CTAs of a pair
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t crank = (CG == 2) ? cluster_ctarank() : 0u;
  const uint32_t rank = crank & 1u;      // this CTA's place in its pair
  const uint32_t leader = crank & ~1u;   // cluster rank of the pair's leader CTA
  const uint16_t pair_mask = static_cast<uint16_t>(0x3u << leader);
  const int cluster_idx = static_cast<int>(blockIdx.x) / CG;
  const int num_clusters = static_cast<int>(gridDim.x) / CG;

  const uint32_t bar_full = base + L::OFF_BAR;       // full[s]: stage s loaded (leader's copy used)
  const uint32_t bar_empty = bar_full + 8 * STAGES;  // empty[s]: stage s consumed by the MMAs
  const uint32_t bar_tfull = bar_empty + 8 * STAGES; // tmem_full[slot]: accumulator ready
  const uint32_t bar_tempty = bar_tfull + 16;        // tmem_empty[slot]: accumulator drained
  const uint32_t bar_never = bar_tempty + 16;        // nobody arrives (timeout-path test)
  const uint32_t bar_drain = bar_never + 8;          // MMA drain after an abort
  const uint32_t bar_cload = bar_drain + 8;          // c_loaded[w]: epilogue warp w's prior-C tile landed
  const uint32_t bar_clc_full = bar_cload + 8 * L::EPI_WARPS;  // clc_full[s]: CLC response s landed here
  const uint32_t bar_clc_empty = bar_clc_full + 8 * kClcSlots; // clc_empty[s] (leader): response s released
  const uint32_t bar_partner = bar_clc_empty + 8 * kClcSlots;  // partner: the other pair's partial sums are written
  const ClcRing ring{base + L::OFF_CLC, bar_clc_full, CG == 2 ? mapa_shared(bar_clc_empty, leader) : bar_clc_empty};
  constexpr bool clc = CLC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEM_SLOT);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::OFF_ABORT);
  const WaitCtx wctx{abort_flag, p.status, p.wait_limit_ns};

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, L::EPI_WARPS * CG);
    }
    mbar_init(bar_never, 1);
    mbar_init(bar_drain, 1);
    for (int w = 0; w < L::EPI_WARPS; ++w) mbar_init(bar_cload + 8 * w, 1);
    for (int t = 0; t < kClcSlots; ++t) {
      mbar_init(bar_clc_full + 8 * t, 1);
      mbar_init(bar_clc_empty + 8 * t, L::CLC_CONSUMERS);
    }
    mbar_init(bar_partner, PAIRS > 1 ? 32 * L::EPI_WARPS * (PAIRS - 1) : 1);
    *abort_flag = 0u;
    fence_mbarrier_init_cluster();
    // every response slot armed for its first use (re-armed by producer A as it reads them)
    if (clc)
      for (int t = 0; t < kClcSlots; ++t) mbar_arrive_expect_tx(bar_clc_full + 8 * t, 16);
    prefetch_tensormap(&tmap_a);
    prefetch_tensormap(&tmap_b);
    prefetch_tensormap(&tmap_b_half);
    prefetch_tensormap(&tmap_c);
  }
  if (warp == 1) {
    tmem_alloc<CG>(smem_u32(tmem_slot), L::TMEM_COLS);
    tmem_relinquish<CG>();
  }
  tc_fence_before_sync();
  if constexpr (CG == 2) cluster_sync_all(); else __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // Set-up is done: the next kernel may start its own. Every global access below (TMA
  // loads and stores) comes after the previous kernel on the stream has completed.
  pdl_launch_dependents();
  pdl_wait();
  clock_probe_mark(p.probe, 0);

  if (warp == 0 || warp == L::WARP_PROD_B) {
    // ------------------------------------------------------------ TMA producers (A: warp 0, B)
    const bool load_a = warp == 0;
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      const bool issuer = clc && load_a && rank == 0;  // requests the CLC responses
      int it = 0;
      for (int i = cluster_idx < p.num_items ? cluster_idx : -1; i >= 0; ++it) {
        if (issuer && !clc_request<(CG == 2)>(ring, bar_clc_empty, it, wctx, status_code(kRoleProducer, 0x200 + it % kClcSlots))) {
          ok = false;
          break;
        }
        const Bf16Item w = bf16_item(p, i, SWAP);
        const TileCoord tc = tile_coord(w.tile, p.num_m_blocks, p.num_n_blocks, p.group_m);
        const bool half = w.half >= 0;
        // K order of the item: every other wave of items walks K downwards, so it starts on
        // the K blocks the previous wave read last (still in L2). Static schedule: a cluster's
        // item count is the wave number. CLC: the wave is item / co-resident clusters.
        const bool down = p.zigzag && (((clc ? i / p.wave : it) & 1) != 0);
        const int a_row = tc.m_blk * L::TILE_M + static_cast<int>(rank) * L::BLOCK_M;
        const int b_row = tc.n_blk * L::BLOCK_N + (half ? w.half * (L::BLOCK_N / 2) + static_cast<int>(rank) * (L::B_ROWS / 2)
                                                        : static_cast<int>(rank) * L::B_ROWS);
        const CUtensorMap* map_b = half ? &tmap_b_half : &tmap_b;
        const uint32_t atom_bytes = L::A_ATOM_BYTES + (half ? L::B_ATOM_BYTES / 2 : L::B_ATOM_BYTES);
        // Straight-line loop body: this producer's operand, map and row are fixed for the tile,
        // the ring position advances by selects (each taken branch costs the thread cycles).
        const uint32_t dst0 = base + (load_a ? L::OFF_A : L::OFF_B);
        const uint32_t atom_stride = load_a ? L::A_ATOM_BYTES : L::B_ATOM_BYTES;
        const uint32_t stage_stride = load_a ? L::A_BYTES : L::B_BYTES;
        const CUtensorMap* map = load_a ? &tmap_a : map_b;
        const int row = load_a ? a_row : b_row;
        const bool arm = load_a && (CG == 1 || rank == 0);
#pragma unroll 2
        for (int kb = 0; kb < w.kn; ++kb) {
          // K block of this stage
          const int kblk = w.k0 + (down ? w.kn - 1 - kb : kb);
          // swizzle-row columns of this stage that hold any of K (the last block may hold fewer)
          const int atoms = min(ATOMS, (p.K - kblk * L::BLOCK_K + L::ATOM_K - 1) / L::ATOM_K);
          const uint32_t stage_bytes = atom_bytes * static_cast<uint32_t>(atoms);
          // First pass over the ring: parity 1 of a fresh barrier counts as complete.
          if (!wait_phase(bar_empty + 8 * stage, phase ^ 1u, wctx, status_code(kRoleProducer, stage))) {
            ok = false;
            break;
          }
          const uint32_t full = bar_full + 8 * stage;
          const uint32_t dst = dst0 + stage * stage_stride;
          const int x0 = kblk * L::BLOCK_K;
          // The A producer arms the barrier with the stage's bytes (of both CTAs for a pair);
          // the B loads may complete before that arrival, the phase cannot.
          if (arm) mbar_arrive_expect_tx(full, (CG == 2 ? 2u : 1u) * stage_bytes);
          const uint32_t target = CG == 2 ? mapa_shared(full, leader) : full;
          if (atoms == ATOMS) {
#pragma unroll
            for (int a = 0; a < ATOMS; ++a) {
              if constexpr (CG == 1) tma_load_2d(dst + a * atom_stride, map, x0 + a * L::ATOM_K, row, target);
              else tma_load_2d_pair(dst + a * atom_stride, map, x0 + a * L::ATOM_K, row, target);
            }
          } else {
            for (int a = 0; a < atoms; ++a) {
              if constexpr (CG == 1) tma_load_2d(dst + a * atom_stride, map, x0 + a * L::ATOM_K, row, target);
              else tma_load_2d_pair(dst + a * atom_stride, map, x0 + a * L::ATOM_K, row, target);
            }
          }
          stage = stage + 1 == STAGES ? 0u : stage + 1;
          phase = stage == 0 ? phase ^ 1u : phase;
        }
        if (!ok) break;
        // next item: producer A re-arms this CTA's response slot for its next use
        i = clc ? clc_next(ring, it, CG, load_a, !issuer, wctx, status_code(kRoleProducer, 0x300 + it % kClcSlots), ok)
                : (i + num_clusters < p.num_items ? i + num_clusters : -1);
      }
      if (!ok) settle_after_abort();
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (rank == 0 && lane == 0) {
      constexpr uint32_t IDESC_FULL = idesc_bf16(L::TILE_M, L::BLOCK_N);
      constexpr uint32_t IDESC_HALF = idesc_bf16(L::TILE_M, L::BLOCK_N / 2);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      if (p.debug_flags & 1u) ok = wait_phase(bar_never, 0, wctx, status_code(kRoleMma, 0xFFFF));
      int it = 0;
      const uint64_t a_desc0 = umma_desc_sw128(base + L::OFF_A), b_desc0 = umma_desc_sw128(base + L::OFF_B);
      for (int i = cluster_idx < p.num_items ? cluster_idx : -1; i >= 0 && ok; ++it) {
        const Bf16Item w = bf16_item(p, i, SWAP);
        const uint32_t idesc = w.half >= 0 ? IDESC_HALF : IDESC_FULL;
        const uint32_t slot = static_cast<uint32_t>(it) & 1u;
        const uint32_t acc_phase = (static_cast<uint32_t>(it) >> 1) & 1u;
        if (!wait_phase(bar_tempty + 8 * slot, acc_phase ^ 1u, wctx, status_code(kRoleMma, 0x100 + slot))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + slot * L::ACC_COLS;
        const bool down = p.zigzag && (((clc ? i / p.wave : it) & 1) != 0);  // the producer's K order for this item
        // Straight-line loop body: descriptors follow from the ring position, which advances
        // by selects; a full stage issues its MMAs without per-MMA tests (each taken branch
        // costs this thread cycles).
#pragma unroll 2
        for (int kb = 0; kb < w.kn; ++kb) {
          const int kblk = w.k0 + (down ? w.kn - 1 - kb : kb);
          if (!wait_phase(bar_full + 8 * stage, phase, wctx, status_code(kRoleMma, stage))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t a_desc = umma_desc_advance(a_desc0, stage * L::A_BYTES);
          const uint64_t b_desc = umma_desc_advance(b_desc0, stage * L::B_BYTES);
          // MMAs of the swizzle-row columns that hold any of K (all of them but in a ragged last stage)
          const int ksteps = min(L::KSTEPS, (p.K - kblk * L::BLOCK_K + L::ATOM_K - 1) / L::ATOM_K * (L::ATOM_K / L::UMMA_K));
          if (ksteps == L::KSTEPS) {
#pragma unroll
            for (int kk = 0; kk < L::KSTEPS; ++kk) {
              // column kk / 4 of the stage, then 32 bytes per MMA inside its 128-byte swizzle row
              const uint32_t koff_a = (kk / 4) * L::A_ATOM_BYTES + (kk % 4) * L::UMMA_K * 2;
              const uint32_t koff_b = (kk / 4) * L::B_ATOM_BYTES + (kk % 4) * L::UMMA_K * 2;
              mma_f16<CG>(d_tmem, umma_desc_advance(a_desc, koff_a), umma_desc_advance(b_desc, koff_b), idesc,
                          (kb | kk) != 0 ? 1u : 0u);
            }
          } else {
            for (int kk = 0; kk < ksteps; ++kk) {
              const uint32_t koff_a = (kk / 4) * L::A_ATOM_BYTES + (kk % 4) * L::UMMA_K * 2;
              const uint32_t koff_b = (kk / 4) * L::B_ATOM_BYTES + (kk % 4) * L::UMMA_K * 2;
              mma_f16<CG>(d_tmem, umma_desc_advance(a_desc, koff_a), umma_desc_advance(b_desc, koff_b), idesc,
                          (kb | kk) != 0 ? 1u : 0u);
            }
          }
          // Release the stage when these MMAs have read it; never wait here.
          if constexpr (CG == 1) mma_commit_local(bar_empty + 8 * stage);
          else mma_commit_pair_multicast(bar_empty + 8 * stage, pair_mask);
          stage = stage + 1 == STAGES ? 0u : stage + 1;
          phase = stage == 0 ? phase ^ 1u : phase;
        }
        if (!ok) break;
        if constexpr (CG == 1) mma_commit_local(bar_tfull + 8 * slot);
        else mma_commit_pair_multicast(bar_tfull + 8 * slot, pair_mask);
        i = clc ? clc_next(ring, it, CG, false, true, wctx, status_code(kRoleMma, 0x300 + it % kClcSlots), ok)
                : (i + num_clusters < p.num_items ? i + num_clusters : -1);
      }
      if (!ok) {
        // let issued MMAs finish before TMEM is released
        if constexpr (CG == 1) mma_commit_local(bar_drain);
        else mma_commit_pair_multicast(bar_drain, static_cast<uint16_t>(1u << leader));
        wait_phase_slow(bar_drain, 0, wctx, status_code(kRoleMma, 0xFFFE), false);
        settle_after_abort();
      }
    }
    __syncwarp();
  } else if (warp >= 2 && warp < 2 + L::EPI_WARPS) {
    // ------------------------------------------------------------ epilogue
    const uint32_t q = warp & 3u;  // this warp may access TMEM lanes 32q .. 32q+31
    const uint32_t epi = warp - 2u;
    const uint32_t stage_base = base + L::OFF_EPI + epi * L::EPI_BUFS * L::EPI_BUF_BYTES;
    const uint32_t tempty_target = (CG == 2) ? mapa_shared(bar_tempty, leader) : bar_tempty;
    const uint32_t cload = bar_cload + 8 * epi;
    uint32_t cload_phase = 0;
    bool epi_ok = true;
    uint32_t ebuf = 0;
    int it = 0;
    for (int i = cluster_idx < p.num_items ? cluster_idx : -1; i >= 0; ++it) {
      const Bf16Item w = bf16_item(p, i, SWAP);
      const TileCoord tc = tile_coord(w.tile, p.num_m_blocks, p.num_n_blocks, p.group_m);
      const int chunks = (w.half >= 0 ? L::BLOCK_N / 2 : L::BLOCK_N) / 64;
      const uint32_t slot = static_cast<uint32_t>(it) & 1u;
      const uint32_t acc_phase = (static_cast<uint32_t>(it) >> 1) & 1u;
      const int row0 = tc.m_blk * L::TILE_M + static_cast<int>(rank) * L::BLOCK_M + static_cast<int>(q) * 32;
      const int col0 = tc.n_blk * L::BLOCK_N + (w.half > 0 ? L::BLOCK_N / 2 : 0);
      if (!SWAP && p.epi.fused && p.epi.beta != 0.0f && lane == 0 && row0 < p.M) {
        // the prior C of this warp's part of the tile into L2 while the MMAs still run
        for (int c = 0; c < chunks; ++c)
          if (col0 + c * 64 < p.N) tma_prefetch_l2_2d(&tmap_c, col0 + c * 64, row0);
      }
      if (!wait_phase_warp(bar_tfull + 8 * slot, acc_phase, wctx, status_code(kRoleEpilogue, slot))) break;
      tc_fence_after_sync();
      if constexpr (SWAP && PAIRS > 1) {
        // the first pair waits until the other pairs' partial sums are in the workspace
        if (w.split == 0 && !wait_phase_warp(bar_partner, 0, wctx, status_code(kRoleEpilogue, 0x700))) break;
      }
      const uint32_t taddr = tmem_base + ((q * 32u) << 16) + slot * L::ACC_COLS;
      if (row0 < p.M) {
#pragma unroll 1
        for (int c = 0; c < chunks; ++c) {
          const int col = col0 + c * 64;
          if (col >= p.N) break;
          uint32_t lo[32], hi[32];
          tmem_ld_32x32b_x32(taddr + c * 64, lo);
          tmem_ld_32x32b_x32(taddr + c * 64 + 32, hi);
          tmem_ld_wait();
          if constexpr (SWAP && PAIRS > 1) {
            const int row = row0 + static_cast<int>(lane);
            if (w.split >= 1) {
              // pair s >= 1: this row's 64 FP32 partial sums of the chunk to workspace slot s - 1
              if (row < p.M) {
                float4* dst = reinterpret_cast<float4*>(
                    p.ws + (static_cast<size_t>(w.split - 1) * p.M + row) * p.ldw + col);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  dst[j] = make_float4(__uint_as_float(lo[4 * j]), __uint_as_float(lo[4 * j + 1]),
                                       __uint_as_float(lo[4 * j + 2]), __uint_as_float(lo[4 * j + 3]));
                  dst[8 + j] = make_float4(__uint_as_float(hi[4 * j]), __uint_as_float(hi[4 * j + 1]),
                                           __uint_as_float(hi[4 * j + 2]), __uint_as_float(hi[4 * j + 3]));
                }
              }
              continue;
            }
            // the first pair: add the other pairs' partial sums, in split order
            if (row < p.M) {
#pragma unroll 1
              for (int sp = 0; sp < PAIRS - 1; ++sp) {
                const float4* src = reinterpret_cast<const float4*>(
                    p.ws + (static_cast<size_t>(sp) * p.M + row) * p.ldw + col);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const float4 a = src[j], b = src[8 + j];
                lo[4 * j] = __float_as_uint(__uint_as_float(lo[4 * j]) + a.x);
                lo[4 * j + 1] = __float_as_uint(__uint_as_float(lo[4 * j + 1]) + a.y);
                lo[4 * j + 2] = __float_as_uint(__uint_as_float(lo[4 * j + 2]) + a.z);
                lo[4 * j + 3] = __float_as_uint(__uint_as_float(lo[4 * j + 3]) + a.w);
                hi[4 * j] = __float_as_uint(__uint_as_float(hi[4 * j]) + b.x);
                hi[4 * j + 1] = __float_as_uint(__uint_as_float(hi[4 * j + 1]) + b.y);
                hi[4 * j + 2] = __float_as_uint(__uint_as_float(hi[4 * j + 2]) + b.z);
                hi[4 * j + 3] = __float_as_uint(__uint_as_float(hi[4 * j + 3]) + b.w);
                }
              }
            }
          } else if constexpr (SWAP) {
            if (p.splits > 1) {
              // a K split: this row's 64 FP32 partial sums of the chunk to the workspace
              const int row = row0 + static_cast<int>(lane);
              if (row < p.M) {
                float4* dst = reinterpret_cast<float4*>(p.ws + (static_cast<size_t>(w.split) * p.M + row) * p.ldw + col);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  dst[j] = make_float4(__uint_as_float(lo[4 * j]), __uint_as_float(lo[4 * j + 1]),
                                       __uint_as_float(lo[4 * j + 2]), __uint_as_float(lo[4 * j + 3]));
                  dst[8 + j] = make_float4(__uint_as_float(hi[4 * j]), __uint_as_float(hi[4 * j + 1]),
                                           __uint_as_float(hi[4 * j + 2]), __uint_as_float(hi[4 * j + 3]));
                }
              }
              continue;
            }
          }
          const uint32_t buf = stage_base + ebuf * L::EPI_BUF_BYTES;
          if (lane == 0) bulk_wait_group_read<1>();  // the store that last read `buf` is done
          __syncwarp();
          // Row `lane` of the 32 x 64 staging tile, 16-byte chunk j at position j ^ (row % 8):
          // the 128-byte swizzle the C tensor map uses (and bank-conflict free).
          const uint32_t row_addr = buf + lane * 128u;
          uint32_t pk[32];
          if constexpr (SWAP) {
            // columns i and 32 + i of this lane's accumulator row, for the transposed tile
            if (!p.epi.fused) {
#pragma unroll
              for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2_rn(lo[i], hi[i]);
            } else {
              // fused epilogue: this lane is column n = row0 + lane of the caller's C, so its
              // bias is one value; its prior C is column `lane` of the transposed 64 x 32 tile
              // (TMA-loaded into the staging buffer, zeros past the caller's M and N)
              const int n = row0 + static_cast<int>(lane);
              const uint32_t bv = (p.epi.bias != nullptr && n < p.M) ? static_cast<uint32_t>(p.epi.bias[n]) : 0u;
              const uint32_t bias2 = bv | (bv << 16);
              const bool with_old = p.epi.beta != 0.0f;
              if (with_old) {
                if (lane == 0) {
                  mbar_arrive_expect_tx(cload, L::EPI_BUF_BYTES);
                  tma_load_2d(buf, &tmap_c, row0, col, cload);  // (column, row) of the caller's C
                }
                if (!wait_phase_warp(cload, cload_phase, wctx, status_code(kRoleEpilogue, 2))) {
                  epi_ok = false;
                  break;
                }
                cload_phase ^= 1u;
              }
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const uint32_t old2 = with_old ? (ld_shared_u16(buf + i * 64 + lane * 2) |
                                                  (ld_shared_u16(buf + (32 + i) * 64 + lane * 2) << 16))
                                               : 0u;
                pk[i] = epi_pair(lo[i], hi[i], old2, bias2, p.epi);
              }
              // every lane has read its column of the prior C before any lane overwrites it
              __syncwarp();
            }
          } else if (!p.epi.fused) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              pk[i] = pack_bf16x2_rn(lo[2 * i], lo[2 * i + 1]);
              pk[16 + i] = pack_bf16x2_rn(hi[2 * i], hi[2 * i + 1]);
            }
          } else {
            // prior C of the chunk (beta != 0): the 32 x 64 tile by TMA into the staging
            // buffer (zeros past M and N), then row `lane` from it
            uint32_t old[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) old[i] = 0u;
            if (p.epi.beta != 0.0f) {
              if (lane == 0) {
                mbar_arrive_expect_tx(cload, L::EPI_BUF_BYTES);
                tma_load_2d(buf, &tmap_c, col, row0, cload);
              }
              if (!wait_phase_warp(cload, cload_phase, wctx, status_code(kRoleEpilogue, 2))) {
                epi_ok = false;
                break;
              }
              cload_phase ^= 1u;
#pragma unroll
              for (int j = 0; j < 8; ++j)
                ld_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4), old[4 * j], old[4 * j + 1],
                             old[4 * j + 2], old[4 * j + 3]);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint4 bb = epi_bias8(p.epi, col + 8 * j, p.N);
              const uint32_t b4[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const int e = 4 * j + t;  // pair index: columns 2e, 2e + 1 of the chunk
                const uint32_t a0 = e < 16 ? lo[2 * e] : hi[2 * e - 32];
                const uint32_t a1 = e < 16 ? lo[2 * e + 1] : hi[2 * e - 31];
                pk[e] = epi_pair(a0, a1, old[e], b4[t], p.epi);
              }
            }
            // every lane has read its row of the prior C before any lane overwrites it
            __syncwarp();
          }
          if constexpr (SWAP) {
            // Transposed staging tile: 64 rows (the chunk's accumulator columns, rows of the
            // caller's C) x 32 BF16 columns (this warp's accumulator rows). For one row, the
            // 32 lanes write 64 consecutive bytes: no bank conflicts.
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              st_shared_u16(buf + i * 64 + lane * 2, static_cast<uint16_t>(pk[i] & 0xFFFFu));
              st_shared_u16(buf + (32 + i) * 64 + lane * 2, static_cast<uint16_t>(pk[i] >> 16));
            }
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4), pk[4 * j], pk[4 * j + 1],
                           pk[4 * j + 2], pk[4 * j + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if constexpr (SWAP) tma_store_2d(&tmap_c, buf, row0, col);  // (column, row) of the caller's C
            else tma_store_2d(&tmap_c, buf, col, row0);
            bulk_commit_group();
          }
          ebuf ^= 1u;
        }
      }
      if constexpr (SWAP && PAIRS > 1) {
        // release this lane's partial sums to the first pair's CTA that holds the same rows
        // (cluster rank 0 or 1: this CTA's place in its pair)
        if (w.split >= 1) mbar_arrive_cluster(mapa_shared(bar_partner, rank));
      }
      if (!epi_ok) break;  // a prior-C load timed out (status recorded)
      // Accumulator slot drained: hand it back to the MMA issuer (leader CTA's barrier).
      tmem_ld_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 2) mbar_arrive_cluster(tempty_target + 8 * slot);
        else mbar_arrive_local(bar_tempty + 8 * slot);
      }
      if (clc) {
        // every lane reads the response; one releases the slot
        const uint32_t s = static_cast<uint32_t>(it) % kClcSlots, ph = (static_cast<uint32_t>(it) / kClcSlots) & 1u;
        if (!wait_phase_warp(ring.full + 8 * s, ph, wctx, status_code(kRoleEpilogue, 0x300 + s))) break;
        uint32_t x;
        const bool got = clc_query(ring.resp + 16 * s, x);
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(ring.empty_leader + 8 * s);
        i = got ? static_cast<int>(x) / CG : -1;
      } else {
        i = i + num_clusters < p.num_items ? i + num_clusters : -1;
      }
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  tc_fence_before_sync();
  if constexpr (CG == 2) cluster_sync_all(); else __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc<CG>(tmem_base, L::TMEM_COLS);
  }
  clock_probe_mark(p.probe, 1);
}

// ---------------------------------------------------------------------------- host side

namespace {

// Split-K reduction of the swapped GEMM: C[m][n] = bf16_rne(sum over s of ws[s][n][m]), C
// being the caller's rows x cols BF16 matrix and ws[s] its transpose (cols rows of ldw
// FP32 values). 32 x 32 tiles through shared memory: reads along m, writes along n. Every
// thread issues all of its loads (4 rows x up to kMaxSplits splits) before the first add,
// so they overlap instead of each waiting for the previous one. Launched with
// programmatic stream serialization: its blocks start while the GEMM drains and wait for
// it (griddepcontrol.wait) before the first read.
constexpr int kMaxSplits = 8;

__global__ void __launch_bounds__(256) splitk_reduce_transposed(const float* __restrict__ ws, uint16_t* __restrict__ C,
                                                                int rows, int cols, int splits, int ldw, EpiParams epi) {
  __shared__ float t[32][33];
  pdl_launch_dependents();
  pdl_wait();
  const int n0 = blockIdx.x * 32, m0 = blockIdx.y * 32;
  const int m = m0 + static_cast<int>(threadIdx.x);
  float v[4][kMaxSplits];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int n = n0 + static_cast<int>(threadIdx.y) + 8 * i;
    const bool in = n < cols && m < rows;
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s)
      v[i][s] = (in && s < splits) ? __ldg(ws + (static_cast<size_t>(s) * cols + n) * ldw + m) : 0.0f;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float acc = 0.0f;
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) acc += v[i][s];  // in split order, as before
    t[threadIdx.y + 8 * i][threadIdx.x] = acc;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += 8) {
    const int mm = m0 + r, n = n0 + static_cast<int>(threadIdx.x);
    if (mm < rows && n < cols) {
      uint16_t* c = C + static_cast<size_t>(mm) * cols + n;
      if (!epi.fused) {
        *c = __bfloat16_as_ushort(__float2bfloat16_rn(t[threadIdx.x][r]));
      } else {
        // the fused epilogue on one value: the pair arithmetic of the GEMM epilogues, low half
        const uint32_t old = epi.beta != 0.0f ? static_cast<uint32_t>(*c) : 0u;
        const uint32_t bias = epi.bias != nullptr ? static_cast<uint32_t>(epi.bias[n]) : 0u;
        *c = static_cast<uint16_t>(epi_pair(__float_as_uint(t[threadIdx.x][r]), 0u, old, bias, epi) & 0xFFFFu);
      }
    }
  }
}

int launch_splitk_reduce(const float* ws, void* C, int rows, int cols, int splits, int ldw, const EpiParams& epi,
                         cudaStream_t stream, int pdl) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(cols, 32)), static_cast<unsigned>(ceil_div(rows, 32)), 1);
  cfg.blockDim = dim3(32, 8, 1);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, splitk_reduce_transposed, ws, static_cast<uint16_t*>(C), rows, cols, splits, ldw, epi) !=
      cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  count_launch();
  return GEMM_OK;
}

template <int CG, int STAGES, int ATOMS, int BN = 256, bool SWAP = false, int PAIRS = 1>
struct Bf16Variant {
  using L = Bf16Layout<CG, STAGES, ATOMS, BN, SWAP>;
  static constexpr int CLUSTER = CG * PAIRS;  // CTAs per cluster
  static constexpr auto kernel = bf16_gemm_kernel<CG, STAGES, ATOMS, BN, SWAP, false, PAIRS>;
  // (two pairs per cluster never use CLC: the same instantiation stands in)
  static constexpr auto kernel_clc = bf16_gemm_kernel<CG, STAGES, ATOMS, BN, SWAP, PAIRS == 1, PAIRS>;

  // Co-resident clusters per device, queried once per device.
  static int max_active_clusters(int device) {
    static std::mutex mu;
    static int cache[64] = {0};
    std::lock_guard<std::mutex> lock(mu);
    if (device < 0 || device >= 64) return 0;
    if (cache[device] > 0) return cache[device];
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(kernel_clc, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_BYTES) != cudaSuccess)
      return 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(CLUSTER * 16, 1, 1);
    cfg.blockDim = dim3(L::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM_BYTES;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CLUSTER;
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

  static int run(const void* A, const void* B, void* C, int M, int N, int K, cudaStream_t stream,
                 const RunOptions& opt, int device, const DeviceInfo& info) {
    CUtensorMap ta, tb, tbh, tc;
    int st = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, K, M, uint64_t(K) * 2, L::ATOM_K,
                            L::BLOCK_M, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == GEMM_OK)
      st = encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, K, N, uint64_t(K) * 2, L::ATOM_K, L::B_ROWS,
                          CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == GEMM_OK)  // B box of a half-width work item
      st = encode_tmap_2d(&tbh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, K, N, uint64_t(K) * 2, L::ATOM_K,
                          L::B_ROWS / 2, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == GEMM_OK) {
      if constexpr (SWAP)  // the caller's C is N x M here: boxes of 64 of its rows x 32 columns
        st = encode_tmap_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, C, M, N, uint64_t(M) * 2, 32, 64,
                            CU_TENSOR_MAP_SWIZZLE_NONE);
      else
        st = encode_tmap_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, C, N, M, uint64_t(N) * 2, 64, 32,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (st != GEMM_OK) return st;

    Bf16Params p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.num_m_blocks = ceil_div(M, L::TILE_M);
    p.num_n_blocks = ceil_div(N, L::BLOCK_N);
    const long long tiles = static_cast<long long>(p.num_m_blocks) * p.num_n_blocks;
    if (tiles > 0x7FFFFFFFLL) return GEMM_ERR_UNSUPPORTED_SHAPE;
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

    const int max_clusters = max_active_clusters(device);
    if (max_clusters <= 0) return GEMM_ERR_LAUNCH;
    // Persistent grid: at most the co-resident clusters. The last partial wave is cut
    // into N-halves when they still fit in one wave.
    int wave = p.num_tiles;
    if (opt.persistent) {
      wave = max_clusters;
      if (opt.max_clusters > 0) wave = std::min(wave, opt.max_clusters);
    }
    // (swapped variants keep whole tiles: their tile N is already small)
    p.split_tiles = (opt.persistent && opt.tail_split && !SWAP) ? tail_split_tiles(p.num_tiles, wave) : 0;
    // K splits (swapped variants): enough work items to occupy the free clusters. A split
    // costs about 4 us (FP32 partials out and back, the reduction kernel), so two splits pay
    // only where halving the per-pair stream saves more: tile N 64 and at least 48 stages
    // (measured at N = K = 8192: 34.1 -> 31.2 us for M = 64; tile N 128 and K = 2048 lost).
    int splits = 1;
    if (SWAP && opt.persistent && opt.split_k) {
      splits = std::min(std::min(wave / std::max(p.num_tiles, 1), kMaxSplits), p.k_iters / 4);
      const bool two_pay = BN == 64 && p.k_iters >= 48;
      if (splits < 2 || (splits == 2 && !two_pay)) splits = 1;
    }
    if constexpr (SWAP && PAIRS == 1 && CG == 2 && BN == 64) {
      // Two splits: one cluster of two pairs per tile adds the halves itself (no second
      // kernel), when enough clusters of four CTAs fit for all tiles at once. (Four pairs
      // per cluster for four splits measured slower than the reduction kernel: 18.1 against
      // 12.8 us at M = 100, N = K = 2048.)
      if (opt.clc != 1 && opt.max_clusters == 0 && splits == 2) {
        using Two = Bf16Variant<CG, STAGES, ATOMS, BN, SWAP, 2>;
        if (Two::max_active_clusters(device) >= p.num_tiles) return Two::run(A, B, C, M, N, K, stream, opt, device, info);
      }
    }
    if constexpr (PAIRS > 1) splits = PAIRS;
    p.k_per_split = ceil_div(p.k_iters, splits);
    p.splits = ceil_div(p.k_iters, p.k_per_split);  // no empty split
    if (PAIRS > 1 && p.splits != PAIRS) return GEMM_ERR_UNSUPPORTED_SHAPE;  // (the split rule rules it out)
    p.ldw = p.num_n_blocks * L::BLOCK_N;
    p.ws = nullptr;
    p.num_items = p.splits > 1 ? p.num_tiles * p.splits : p.num_tiles + p.split_tiles;
    // Cluster launch control: the whole grid of one cluster per item, taken dynamically
    p.clc = (PAIRS == 1 && opt.persistent && opt.max_clusters == 0 && use_clc(opt.clc, p.num_items, max_clusters, K, false)) ? 1 : 0;
    // (two pairs per cluster: every pair computes exactly one item)
    const int clusters = (p.clc || PAIRS > 1) ? p.num_items : std::min(p.num_items, wave);
    p.wave = std::max(wave, 1);
    p.group_m = opt.group_m > 0 ? std::min(opt.group_m, p.num_m_blocks)
                                : choose_group_m(M, N, K, L::TILE_M, L::BLOCK_N, 2.0, 0.0, clusters, info.l2_bytes);

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * CG), 1, 1);
    cfg.blockDim = dim3(L::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM_BYTES;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CLUSTER;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = opt.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (p.splits > 1) {
      // FP32 partials of every split, from the library's stream-ordered pool
      cudaMemPool_t pool = workspace_pool(device);
      void* ws = nullptr;
      // (several pairs per cluster: the first pair's part never goes through the workspace)
      const size_t bytes = static_cast<size_t>(PAIRS > 1 ? PAIRS - 1 : p.splits) * p.M * p.ldw * sizeof(float);
      if (pool == nullptr || cudaMallocFromPoolAsync(&ws, bytes, pool, stream) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_OUT_OF_MEMORY;
      }
      p.ws = static_cast<float*>(ws);
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, p.clc ? kernel_clc : kernel, ta, tb, tbh, tc, p);
    int st2 = GEMM_OK;
    if (e != cudaSuccess) {
      cudaGetLastError();
      st2 = GEMM_ERR_LAUNCH;
    } else {
      count_launch();
    }
    if (p.splits > 1) {
      if (PAIRS == 1 && st2 == GEMM_OK)
        st2 = launch_splitk_reduce(p.ws, C, p.N, p.M, p.splits, p.ldw, p.epi, stream, opt.pdl);
      if (cudaFreeAsync(p.ws, stream) != cudaSuccess && st2 == GEMM_OK) st2 = GEMM_ERR_LAUNCH;
    }
    return st2;
  }
};

using Bf16OneCta = Bf16Variant<1, 4, 1>;
using Bf16Pair = Bf16Variant<2, 3, 2>;     // 3 stages of 128 K (64 KB per CTA): the default
using Bf16PairK64 = Bf16Variant<2, 6, 1>;  // 6 stages of 64 K (32 KB per CTA)
// C^T = B A^T for M <= 64 / M <= 128: tile N 64 / 128, 4 stages of 128 K (40 / 48 KB per CTA)
using Bf16Swap64 = Bf16Variant<2, 4, 2, 64, true>;
using Bf16Swap128 = Bf16Variant<2, 4, 2, 128, true>;

}  // namespace

// A GEMM with few rows wastes most of each M = 256 MMA on padding; computed as C^T = B A^T
// its rows become the MMA's N (64 or 128) and the long N dimension fills the 256 MMA rows.
bool bf16_swap_ab(int M, int N, const RunOptions& opt) {
  return opt.swap_ab && opt.kernel == GEMM_KERNEL_DEFAULT && M >= 1 && M <= 128 && N >= 256;
}

// The default kernel for a GEMM that is not swapped: the 512 x 256 pair tile where
// wide_rule favours it, with a static schedule (cluster launch control, when asked for,
// runs on the 256 x 256 kernel).
bool bf16_use_wide(int M, int N, int K, const RunOptions& opt, int wave) {
  if (opt.kernel != GEMM_KERNEL_DEFAULT || !opt.persistent || opt.max_clusters > 0) return false;
  if (bf16_swap_ab(M, N, opt)) return false;
  if (opt.clc == 1) return false;
  return wide_rule(M, N, K, wave);
}

int bf16_tile_n(int M, int N, const RunOptions& opt) {
  if (!bf16_swap_ab(M, N, opt)) return opt.kernel == GEMM_KERNEL_BF16_1CTA ? Bf16OneCta::L::BLOCK_N : Bf16Pair::L::BLOCK_N;
  return M <= 64 ? Bf16Swap64::L::BLOCK_N : Bf16Swap128::L::BLOCK_N;
}

int run_gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K, cudaStream_t stream,
                  const RunOptions& opt) {
  int device = 0, err = 0;
  const DeviceInfo* info = current_device_info(&device, &err);
  if (info == nullptr) return err;
  switch (opt.kernel) {
    case GEMM_KERNEL_BF16_1CTA:
      return Bf16OneCta::run(A, B, C, M, N, K, stream, opt, device, *info);
    case GEMM_KERNEL_DEFAULT:
      if (bf16_swap_ab(M, N, opt)) {
        if (M <= 64) return Bf16Swap64::run(B, A, C, N, M, K, stream, opt, device, *info);
        return Bf16Swap128::run(B, A, C, N, M, K, stream, opt, device, *info);
      }
      if (bf16_use_wide(M, N, K, opt, Bf16Pair::max_active_clusters(device)))
        return run_gemm_bf16_wide(A, B, C, M, N, K, stream, opt);
      return Bf16Pair::run(A, B, C, M, N, K, stream, opt, device, *info);
    case GEMM_KERNEL_BF16_2CTA:
      return Bf16Pair::run(A, B, C, M, N, K, stream, opt, device, *info);
    case GEMM_KERNEL_BF16_2CTA_K64:
      return Bf16PairK64::run(A, B, C, M, N, K, stream, opt, device, *info);
    case GEMM_KERNEL_BF16_2CTA_WIDE:
      return run_gemm_bf16_wide(A, B, C, M, N, K, stream, opt);
    default:
      return GEMM_ERR_INVALID_ARG;
  }
}

}  // namespace dtcp

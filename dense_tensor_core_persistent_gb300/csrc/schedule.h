// schedule.h -- persistent tile order, shared by the kernels (device) and the host
// helpers/tests (gemm_tile_coord, gemm_choose_group_m).
//
// Output tiles are walked M-first inside groups of `group_m` consecutive M-blocks,
// one group after another; the last group may be shorter. Consecutive tiles (those a
// wave of co-resident clusters works on together) then share a few B tiles and a few A
// tiles, so the operands are re-read from L2 rather than from HBM.
// ("Achieve cuBLAS Performance on NVIDIA GB300 for HGEMM", v6: tile-swizzle scheduling
// walks M-tiles first within groups of SWIZZLE_GROUP; "NVFP4 GEMM on Blackwell",
// Kernel 5: supergroup ordering for L2 reuse.)
#pragma once

#if defined(__CUDACC__)
#define DTCP_HD __host__ __device__ __forceinline__
#else
#define DTCP_HD inline
#endif

namespace dtcp {

struct TileCoord {
  int m_blk;
  int n_blk;
};

// a >= 0, b > 0; no intermediate exceeds a, so a near INT_MAX does not overflow.
DTCP_HD int ceil_div(int a, int b) { return a / b + (a % b != 0 ? 1 : 0); }

// Tile index t (0 <= t < num_m * num_n) -> block coordinates. Requires 1 <= group_m.
DTCP_HD TileCoord tile_coord(int t, int num_m, int num_n, int group_m) {
  if (group_m > num_m) group_m = num_m;
  const int per_group = group_m * num_n;       // tiles in one full group
  const int g = t / per_group;
  const int first_m = g * group_m;
  const int rows = (num_m - first_m < group_m) ? (num_m - first_m) : group_m;
  const int local = t - g * per_group;
  TileCoord c;
  c.m_blk = first_m + local % rows;
  c.n_blk = local / rows;
  return c;
}

// Work items of a persistent launch: the tiles in schedule order, except that the last
// `split_tiles` tiles are each cut into two halves along N. The halves form the final
// partial wave, which then occupies twice as many clusters for half as long.
struct WorkItem {
  int tile;
  int half;  // -1: the whole tile; 0 / 1: the lower / upper half of its columns
};

DTCP_HD WorkItem work_item(int i, int num_tiles, int split_tiles) {
  const int whole = num_tiles - split_tiles;
  WorkItem w;
  if (i < whole) {
    w.tile = i;
    w.half = -1;
  } else {
    const int j = i - whole;
    w.tile = whole + (j >> 1);
    w.half = j & 1;
  }
  return w;
}

// How many trailing tiles to split for a grid of `clusters` co-resident clusters: the
// last wave's tiles, when their halves still fit in one wave.
DTCP_HD int tail_split_tiles(int num_tiles, int clusters) {
  if (clusters <= 1 || num_tiles <= 0) return 0;
  const int tail = num_tiles % clusters;
  return (tail > 0 && 2 * tail <= clusters) ? tail : 0;
}

// Whether a persistent launch of `items` work items, with `wave` co-resident clusters and
// depth K, schedules them dynamically with cluster launch control (CLC) rather than by a
// fixed grid stride. Within one wave there is nothing to balance. Beyond it, measured on
// GB300 (2304 to 16384 on a side): both orders run the same items at the same time, but
// the dynamic one changes which SM pair computes which tile of a wave, and the launch then
// reads up to 2.8x as many bytes from DRAM. For BF16 that costs 3-14% with K up to 12288
// (also at 4 to 54 waves), while with K = 16384 or more the dynamic order gains 0.6-2%.
// For NVFP4 it gained nowhere beyond noise (K = 32768 at 4096^2: 0.5%) and lost up to 13%
// (16384^3), so NVFP4 keeps the static order. ("NVFP4 GEMM on Blackwell", static vs dynamic
// tile scheduling, settled on CLC from four waves on and, for one to four waves, only for
// K >= 16384, for another kernel on another GPU.)
DTCP_HD bool clc_rule(int items, int wave, int K, bool nvfp4) { return !nvfp4 && items > wave && K >= 16384; }

// Tile-times a static persistent launch of `tiles` equal tiles takes on `wave` co-resident
// clusters: its full waves, plus a last partial wave that runs either as whole tiles (one
// tile-time) or, when its tiles' N-halves fit in one wave (tail_split_tiles), as halves,
// which take about 0.8 of a tile's time (measured on GB300 for BF16: an N = 128 MMA costs
// the issuing thread nearly as much as an N = 256 one).
inline double launch_tile_times(long long tiles, long long wave) {
  if (tiles <= 0 || wave <= 0) return 0.0;
  const long long full = tiles / wave, tail = tiles % wave;
  if (tail == 0) return static_cast<double>(full);
  return static_cast<double>(full) + ((wave > 1 && 2 * tail <= wave) ? 0.8 : 1.0);
}

// Whether a plain BF16 GEMM runs on the 512 x 256 pair tile (two 128-row M-waves per CTA)
// rather than the 256 x 256 one, with `wave` co-resident clusters of either. The wide tile
// moves a quarter fewer bytes from L2 per FLOP and keeps one more stage in flight, but has
// half as many tiles to spread over the clusters and one accumulator (its tile boundary
// waits for the epilogue to read TMEM). So: K >= 2048, and the estimated time in
// tile-times is lower, a wide tile counting 2 / f of a 256 x 256 one. f is what a wide
// tile gained per unit of work in sustained runs on GB300 (under the 1.4 kW power cap,
// where its smaller data movement also buys clock): 1.035 at K = 2048 (8192^2 x 2048),
// 1.05-1.08 from K = 4096 (4096^3, 2048 x 8192^2, 3072^2 x 8192, 16384 x 8192^2), so
// f = 1.03 below K = 4096 and 1.06 from there.
inline bool wide_rule(int M, int N, int K, int wave) {
  if (K < 2048 || wave < 1 || M < 1 || N < 1) return false;
  const double f = K < 4096 ? 1.03 : 1.06;
  const long long nb = (N + 255) / 256;
  const long long tiles_std = static_cast<long long>((M + 255) / 256) * nb;
  const long long tiles_wide = static_cast<long long>((M + 511) / 512) * nb;
  return 2.0 * launch_tile_times(tiles_wide, wave) / f < launch_tile_times(tiles_std, wave);
}

// mode: 0 = clc_rule, 1 = always, 2 = never.
DTCP_HD bool use_clc(int mode, int items, int wave, int K, bool nvfp4) {
  return mode == 1 ? true : (mode == 2 ? false : clc_rule(items, wave, K, nvfp4));
}

}  // namespace dtcp

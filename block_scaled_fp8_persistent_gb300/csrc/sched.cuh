// Grouped persistent tile scheduler (device side).
//
// Tiles are numbered expert by expert; inside expert e there are ceil(M_e / BM) row
// tiles times N / BN column tiles, walked in bands of BAND row tiles: inside a band the row
// index is fastest, so the tiles in flight at one time share a few columns of B (read from
// DRAM once per band instead of once per wave) while the band's rows of A stay in L2 as
// its columns go by.  BAND = 1 is the plain order, column index fastest.  A persistent CTA
// takes tiles
// blockIdx.x, blockIdx.x + gridDim.x, ... (the static stride of the SpsTileScheduler in
// the Triton Gluon example "Overlapping Accumulator Block-Scaled Matrix Multiplication",
// Partitions section), and maps a tile id to (expert, first row, first column) by walking
// the expert row offsets forward -- the ids a CTA visits only grow, so each role keeps a
// cursor and the walk costs O(E + tiles) per CTA without any table in memory.  Experts
// with no rows own no tiles, and so do groups whose row count lies outside the launch's
// [min_group_rows, max_group_rows) (two launches of different tile forms split the groups
// by size).  Row segments are groups; group g multiplies the weights (B
// rows and B scales) of expert expert_ids[g], the mapping from group index to expert rows of
// B in promote_accumulators (MAX kernels, grouped_matmul_sm100_blockwise_fp8, Args); without
// an expert_ids array group g uses expert g.
#pragma once
#include <cstdint>
#include "common.cuh"
#include "ptx.cuh"

namespace bsfp8 {

struct TileCoord {
  int e;           // group (row segment)
  int be;          // expert whose weights the group multiplies (rows of B and B scales)
  int64_t m0;      // first row of the tile (global row index)
  int n0;          // first column of the tile
  int64_t m_end;   // one past the expert's last row (rows >= m_end are not this tile's)
};

template <int BM, int BN, int BAND = 1>
struct GroupedScheduler {
  // Only the cursor lives here; offsets, expert ids, group count and N are read from the
  // kernel's parameter block (constant memory) at each call, so they cost no registers.
  int e = -1;           // current group (-1 before the first locate)
  int be = 0;           // its expert
  int64_t base = 0;     // id of the first tile of group e
  int64_t e_tiles = 0;  // tiles of group e
  int64_t r0 = 0, r1 = 0;  // rows of group e
  int64_t rt = 0;          // row tiles of group e

  // t must not decrease between calls.  Returns false past the last tile.  Args has
  // offsets [E+1], expert_ids [E] (or nullptr), E (groups), N and the group row range.
  template <class Args>
  __device__ bool locate(const Args& a, int64_t t, TileCoord& c) {
    const int n_tiles = (a.N + BN - 1) / BN;  // the last column tile may be partial
    while (t >= base + e_tiles) {
      base += e_tiles;
      ++e;
      if (e >= a.E) return false;
      r0 = ldg_s32(a.offsets + e);
      r1 = ldg_s32(a.offsets + e + 1);
      const int64_t rows = r1 - r0;
      rt = (rows >= a.min_group_rows && rows < a.max_group_rows) ? (rows + BM - 1) / BM : 0;
      e_tiles = rt * (int64_t)n_tiles;
      be = a.expert_ids ? ldg_s32(a.expert_ids + e) : e;
    }
    const int64_t local = t - base;
    const int64_t band = local / ((int64_t)BAND * n_tiles);
    const int64_t in_band = local - band * BAND * n_tiles;
    const int64_t band_rows = rt - band * BAND < BAND ? rt - band * BAND : BAND;
    c.e = e;
    c.be = be;
    c.m0 = r0 + (band * BAND + in_band % band_rows) * BM;
    c.n0 = (int)(in_band / band_rows) * BN;
    c.m_end = r1;
    if constexpr (BSFP8_DEBUG) {
      const bool inside = c.m0 >= r0 && c.m0 < r1 && r1 <= a.M_total && c.n0 >= 0 &&
                          c.n0 < a.N && c.be >= 0 && c.be < a.num_experts;
      if (!inside) {
        atomicCAS(a.err, 0, (int)DEV_BOUNDS);
        return false;
      }
    }
    return true;
  }
};

// Validate the group offsets (and the expert ids, when given) and count the row tiles (sum
// over the groups with min_rows <= M_g < max_rows of ceil(M_g / BM)).  Executed by one full
// warp; every lane gets the results: status 0, or the device error code (bad_offsets_code /
// bad_ids_code) to report.
template <int BM>
__device__ __forceinline__ void validate_offsets(const int32_t* off, const int32_t* ids, int E,
                                                 int num_experts, int64_t M_total,
                                                 int64_t min_rows, int64_t max_rows,
                                                 int bad_offsets_code, int bad_ids_code,
                                                 int& status, int64_t& row_tiles) {
  const uint32_t lane = lane_id();
  int good = 1, good_ids = 1;
  long long tiles = 0;
  for (int e = (int)lane; e < E; e += 32) {
    const int a = ldg_s32(off + e), b = ldg_s32(off + e + 1);
    if (b < a) good = 0;
    else if (b - a >= min_rows && b - a < max_rows) tiles += (b - a + BM - 1) / BM;
    if (ids) {
      const int x = ldg_s32(ids + e);
      if (x < 0 || x >= num_experts) good_ids = 0;
    }
  }
  if (lane == 0 && (ldg_s32(off) != 0 || (int64_t)ldg_s32(off + E) != M_total)) good = 0;
  for (int s = 16; s > 0; s >>= 1) tiles += __shfl_xor_sync(0xffffffffu, tiles, s);
  status = !__all_sync(0xffffffffu, good)       ? bad_offsets_code
           : !__all_sync(0xffffffffu, good_ids) ? bad_ids_code
                                                : 0;
  row_tiles = tiles;
}

}  // namespace bsfp8

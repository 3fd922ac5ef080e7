// Grouped persistent tile scheduler (device side).
//
// Tiles are numbered expert by expert; inside expert e there are ceil(M_e / BM) row
// tiles times N / BN column tiles, column index fastest.  A persistent CTA takes tiles
// blockIdx.x, blockIdx.x + gridDim.x, ... (the static stride of the SpsTileScheduler in
// the Triton Gluon example "Overlapping Accumulator Block-Scaled Matrix Multiplication",
// Partitions section), and maps a tile id to (expert, first row, first column) by walking
// the expert row offsets forward -- the ids a CTA visits only grow, so each role keeps a
// cursor and the walk costs O(E + tiles) per CTA without any table in memory.  Experts
// with no rows own no tiles.  The expert -> B rows mapping is the identity (group e uses
// expert e's weights), the reading of expert_ids in promote_accumulators (MAX kernels,
// grouped_matmul_sm100_blockwise_fp8, Args).
#pragma once
#include <cstdint>
#include "ptx.cuh"

namespace bsfp8 {

struct TileCoord {
  int e;           // expert
  int64_t m0;      // first row of the tile (global row index)
  int n0;          // first column of the tile
  int64_t m_end;   // one past the expert's last row (rows >= m_end are not this tile's)
};

template <int BM, int BN>
struct GroupedScheduler {
  const int32_t* off;
  int E;
  int n_tiles;      // ceil(N / BN); the last column tile may be partial
  int e;            // current expert (-1 before the first locate)
  int64_t base;     // id of the first tile of expert e
  int64_t e_tiles;  // tiles of expert e
  int64_t r0, r1;   // rows of expert e

  __device__ GroupedScheduler(const int32_t* offsets, int num_experts, int N)
      : off(offsets), E(num_experts), n_tiles((N + BN - 1) / BN), e(-1), base(0), e_tiles(0), r0(0), r1(0) {}

  // t must not decrease between calls.  Returns false past the last tile.
  __device__ bool locate(int64_t t, TileCoord& c) {
    while (t >= base + e_tiles) {
      base += e_tiles;
      ++e;
      if (e >= E) return false;
      r0 = ldg_s32(off + e);
      r1 = ldg_s32(off + e + 1);
      e_tiles = ((r1 - r0 + BM - 1) / BM) * (int64_t)n_tiles;
    }
    const int64_t local = t - base;
    c.e = e;
    c.m0 = r0 + (local / n_tiles) * BM;
    c.n0 = (int)(local % n_tiles) * BN;
    c.m_end = r1;
    return true;
  }
};

// Validate the offsets and count the row tiles (sum over experts of ceil(M_e / BM)).
// Executed by one full warp; every lane gets the results.
template <int BM>
__device__ __forceinline__ void validate_offsets(const int32_t* off, int E, int64_t M_total,
                                                 int& ok, int64_t& row_tiles) {
  const uint32_t lane = lane_id();
  int good = 1;
  long long tiles = 0;
  for (int e = (int)lane; e < E; e += 32) {
    const int a = ldg_s32(off + e), b = ldg_s32(off + e + 1);
    if (b < a) good = 0;
    else tiles += (b - a + BM - 1) / BM;
  }
  if (lane == 0 && (ldg_s32(off) != 0 || (int64_t)ldg_s32(off + E) != M_total)) good = 0;
  for (int s = 16; s > 0; s >>= 1) tiles += __shfl_xor_sync(0xffffffffu, tiles, s);
  ok = __all_sync(0xffffffffu, good);
  row_tiles = tiles;
}

}  // namespace bsfp8

// TMEM storage plan for double-buffered block-scaled accumulators.
//
// A 2-CTA block-scaled MMA tile of BLOCK_N = 256 fp32 columns needs, per CTA, the
// accumulator plus the scale columns the MMA reads (A scales: BLOCK_K / VEC columns; B
// scales: that many per 128-column block of N).  Two 256-column accumulators fill all 512
// TMEM columns, so the second one is shifted left by exactly the scale columns: it overlaps
// the first in that many columns, and the scales live in the freed columns at the top.
// The epilogue drains the overlapped columns first and releases them early so the next
// tile's MMA can start.  (Overlapping Accumulator Layout section and
// tmem_overlap_storage_plan of the Triton Gluon example "Overlapping Accumulator
// Block-Scaled Matrix Multiplication".)
#pragma once

namespace bsfp8 {

struct TmemPlan {
  int left_offset, left_cols;    // accumulator of even tiles
  int right_offset, right_cols;  // accumulator of odd tiles
  int a_scale_offset, a_scale_cols;
  int b_scale_offset, b_scale_cols;
  int early_release_subtile;     // epilogue subtile (in drain order) holding the overlap
};

__host__ __device__ constexpr TmemPlan tmem_overlap_plan(int block_k, int epilogue_n, int vec,
                                                         bool overlap, int block_n = 256,
                                                         int tmem_cols = 512) {
  // one scale column per VEC elements of K; B scales once per 128-column block of N
  const int a_cols = block_k / vec;
  const int b_cols = a_cols * (block_n / 128);
  const int shared = a_cols + b_cols;
  if (!overlap) {  // single accumulator: scales right after it
    return TmemPlan{0, block_n, 0, block_n, block_n, a_cols, block_n + a_cols, b_cols, 0};
  }
  return TmemPlan{0,
                  block_n,
                  block_n - shared,       // right accumulator starts below the end of left
                  block_n,
                  tmem_cols - shared,     // scales fill the top columns
                  a_cols,
                  tmem_cols - shared + a_cols,
                  b_cols,
                  (shared - 1) / epilogue_n};
}

}  // namespace bsfp8

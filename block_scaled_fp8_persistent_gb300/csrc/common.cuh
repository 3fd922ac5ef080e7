// Types shared by the C-ABI layer (capi.cu) and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "tmem_plan.cuh"

namespace bsfp8 {

// Device-side error codes (written once per launch into the library's error word).
enum DeviceError : int {
  DEV_OK = 0,
  DEV_BAD_OFFSETS = 6,  // offsets[0] != 0, offsets[E] != M_total or not non-decreasing
  DEV_TIMEOUT = 7,      // a pipeline wait gave up (the kernel wound down cleanly)
  DEV_BAD_EXPERT_IDS = 8,  // an expert id outside [0, num_experts)
  DEV_BOUNDS = 10,  // debug builds: a tile's rows, columns or expert fell outside the problem
};

// Debug builds (-DBSFP8_DEBUG=1) check every tile's coordinates against the problem before
// any role uses them (GroupedScheduler::locate): a tile outside it records DEV_BOUNDS and
// ends the kernel's tile walk in every role at once, instead of touching memory out of
// range.  Release builds compile the checks away.
#ifndef BSFP8_DEBUG
#define BSFP8_DEBUG 0
#endif

// Plain pointers and sizes handed to every kernel (tensor maps travel separately as
// __grid_constant__ parameters).
struct GemmArgs {
  const int32_t* offsets;  // [E+1] row offsets per expert
  const void* a_scales;    // blockwise: f32 [K/128, M_total]   MX: u8 [M_total, K/32]
  const void* b_scales;    // blockwise: f32 [E, N/128, K/128]  MX: u8 [E, N, K/32]
  void* C;                 // bf16 [M_total, N]
  int64_t M_total;
  int N, K;
  int E;                   // groups (row segments of A): offsets has E+1 entries
  int* err;                // library-owned device error word
  const int32_t* expert_ids;  // [E] group -> expert (rows of B and B scales); nullptr: identity
  int num_experts;         // experts in B (bound of expert_ids)
  int b_scales_packed;     // MX swap-AB kernel: b_scales in the 512-byte block layout
  // Groups this launch computes: those with min_group_rows <= rows < max_group_rows (the
  // others own no tiles here; a second launch with the complementary range takes them).
  int64_t min_group_rows = 0;
  int64_t max_group_rows = INT64_MAX;
};

// Tile configurations of the blockwise kernel.
enum BlockwiseTile : int {
  TILE_CTA1_256 = 0,  // one CTA, 128 x 256 tile
  TILE_PAIR_256 = 1,  // CTA pair, 256 x 256 tile
  TILE_PAIR_160 = 2,  // CTA pair, 256 x 160 tile, 3-deep TMEM ring
  TILE_PAIR_128 = 3,  // CTA pair, 256 x 128 tile, 4-deep TMEM ring
  TILE_CTA1_128 = 4,  // one CTA, 128 x 128 tile, 4-deep TMEM ring
  TILE_CTA1_96 = 5,   // one CTA, 96 x 256 tile, role warps on the spare TMEM sub-partition
  TILE_PAIR_192 = 6,  // CTA pair, 192 x 256 tile, the same per CTA
  TILE_CTA1_96x192 = 7,   // one CTA, 96 x 192 tile: each epilogue warp drains its 96 columns at once
  TILE_PAIR_192x192 = 8,  // CTA pair, 192 x 192 tile, the same per CTA
  TILE_CTA1_128x192 = 9,  // one CTA, 128 x 192 tile (12 warps)
  TILE_PAIR_224 = 10,     // CTA pair, 224 x 256 tile: 96-row leader with the role warps, 128-row peer
};

// Rows of B each CTA loads per stage (the B tensor map's box height) for a tile config.
int blockwise_b_rows(BlockwiseTile tile);
// Rows of A each CTA loads per stage (the A tensor map's box height).
int blockwise_a_rows(BlockwiseTile tile);

// Launchers (one per kernel family); return the launch error.
cudaError_t launch_bsfp8_blockwise(BlockwiseTile tile, const CUtensorMap& tmA,
                                   const CUtensorMap& tmB, const GemmArgs& args, int num_sms,
                                   cudaStream_t stream);

// MXFP8 (UE8M0 scales per 32 K) grouped GEMM, swap-AB tiles of 128 weight rows x tn token
// rows; tn is 32, 64 or 128.
cudaError_t launch_bsmxfp8(int tn, const CUtensorMap& tmA, const CUtensorMap& tmB,
                           const GemmArgs& args, int num_sms, cudaStream_t stream);

// The same kernel with packed e2m1 weights (mxfp4) and e4m3 tokens, or packed e2m1 tokens
// too (a_fp4).  mma_kind (a_fp4 only): the packed tiles feed kind::mxf4 as loaded, stage_k
// (128 or 256) K per stage, and tmA / tmB map them with [stage_k/2-byte x rows] boxes swizzled
// over the box width.  stage_k = 256 requires chunkable scale rows: K % 512 == 0 and 16-byte
// aligned scales (b_scales unless pre-packed).  mma_kind with e4m3 tokens: kind::mxf8f6f4 on
// e2m1 weights that tmB loads padded (CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, [128 elements x
// 128 rows] boxes, 128-byte swizzle), tmA as for MXFP8.  Otherwise the tiles are re-encoded
// on chip as e4m3 for kind::mxf8f6f4 and the packed operands are mapped with [64-byte x rows]
// boxes and no swizzle.
cudaError_t launch_bsmxfp4(int tn, bool a_fp4, bool mma_kind, int stage_k, const CUtensorMap& tmA,
                           const CUtensorMap& tmB, const GemmArgs& args, int num_sms,
                           cudaStream_t stream);

// nvfp4 x nvfp4 (packed e2m1, e4m3 scales per 16 K, row-major [rows, K/16]) in the same
// kernel.  mma_kind: kind::mxf4nvf4 with scale_vec::4X on the packed tiles (boxes as above;
// stage_k = 256 requires K % 256 == 0 and 16-byte aligned scales); otherwise the tiles are
// dequantized on chip to fp16 for kind::f16 (boxes without swizzle).
cudaError_t launch_bsnvfp4(int tn, bool mma_kind, int stage_k, const CUtensorMap& tmA,
                           const CUtensorMap& tmB, const GemmArgs& args, int num_sms,
                           cudaStream_t stream);

// MXFP8 grouped GEMM with CTA-pair 256 x 256 tiles and overlapping TMEM accumulators.
cudaError_t launch_bsmxfp8_pair(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                const GemmArgs& args, int num_sms, cudaStream_t stream);
// The same CTA-pair kernel with fp4 operands (fmt: 1 = mxfp8 tokens x mxfp4 weights, tmB a
// padded e2m1 map [128 elements x 128 rows]; 2 = mxfp4 x mxfp4 and 3 = nvfp4 x nvfp4, packed
// maps [128 bytes x 128 rows], K blocks of 256).  The fp4 x fp4 forms need chunkable scale
// rows (K % 512 == 0 for mxfp4, K % 256 for nvfp4; 16-byte aligned scales) and row-major
// weight scales; the host launches them only then.
cudaError_t launch_bsmx_pair_fp4(int fmt, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                 const GemmArgs& args, int num_sms, cudaStream_t stream);
// The TMEM plan that kernel is compiled with.
TmemPlan mx_pair_tmem_plan();

// Rearrange UE8M0 B scales [E, N, K/32] into [E, N/128, K/128] blocks of 512 bytes: row r of
// a 128-row block keeps its 4 codes of the 128-K block at byte (r % 32) * 16 + (r / 32) * 4.
cudaError_t launch_pack_mx_b_scales(const uint8_t* src, uint8_t* dst, int E, int N, int K,
                                    int num_sms, cudaStream_t stream);

}  // namespace bsfp8

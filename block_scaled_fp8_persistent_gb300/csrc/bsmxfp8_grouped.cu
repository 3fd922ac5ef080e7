// MXFP8 grouped GEMM for sm_103a: e4m3 operands with UE8M0 scales per 32 K elements,
// applied by the block-scaled tensor-core MMA.
//
//   C[m, n] = sum_k A[m,k] * B[e,n,k] * 2^(a_scales[m, k/32] - 127) * 2^(b_scales[e, n, k/32] - 127)
//
// Prior art: the Triton Gluon example "Overlapping Accumulator Block-Scaled Matrix
// Multiplication" -- scale tiles copied SMEM -> TMEM with tcgen05_copy in the 4 x 32 x 4
// "packed block" arrangement of swizzle_scales_packed_block / unswizzle_scales_shared_memory,
// then tcgen05_mma_scaled on "e4m3" operands, VEC_SIZE = 32 for uint8 scales; persistent
// static tile stride; load / MMA / epilogue partitions.  Differences: the scales arrive in
// their logical row-major layout and are packed on chip; tiles are grouped by expert; and
// the tile is "swap-AB": the MMA's M operand is 128 rows of the expert's weights B and its
// N operand is the expert's token rows of A (tn = 32 / 64 / 128), which suits the small
// per-expert token counts of decode (the swapAB mode of the TileScheduler in the MAX
// grouped_matmul_sm100_blockwise_fp8 kernels).
//
// fp4 operands (the example's mxfp4 and nvfp4 formats: e2m1 elements packed two per byte
// along K; UE8M0 scales per 32, or e4m3 scales per 16 for nvfp4), both operands fp4: the
// packed tiles feed the fp4 block-scaled MMA kinds as TMA loads them (64-byte rows of 128 K,
// 64-byte swizzle), two K = 64 MMAs per stage -- kind::mxf4 (scale_vec::2X: the scale-factor
// id, 0 or 2, picks the byte pair of the stage's scale word) and kind::mxf4nvf4 with
// scale_vec::4X (unsigned e4m3 scales; each MMA reads a whole word, so a stage has two
// 4-column scale groups per operand).  As the example does for these pairs.
//
// Converting forms (mxfp8 tokens with mxfp4 weights, whose only MMA kind takes K = 32 per
// instruction; and the both-fp4 pairs on request, for comparison).  mxfp4: every e2m1 value
// v is exactly an e4m3 value, and the e4m3 code (sign << 7) | (magnitude code << 2) is
// exactly v * 2^-6 (e2m1's subnormal 0.5 lands on e4m3's subnormal 2^-7, zero on zero).  So
// the kernel loads the packed tiles with TMA, converter warps re-encode them into the
// 128-byte-swizzled e4m3 tile the MMA reads, the MMA and its scales are those of mxfp8, and
// the epilogue multiplies by 2^6 per fp4 operand (exact in fp32).  The result is the mxfp8
// result of the same values as long as the MMA's products, 2^-6 per fp4 operand below the
// true ones, stay in fp32's normal range: true products of magnitude at least 2^-120 (one
// fp4 operand) or 2^-114 (two).  (Folding 2^6 into the token scale codes instead measured
// 6-12 % slower on the decode shape.)  nvfp4: the converters dequantize each packed tile
// with its scales into fp16 (exact: an e2m1 value times an e4m3 scale has at most 6
// significant bits and lies inside the normal fp16 range), and the MMA thread issues
// kind::f16 MMAs (K = 16) with no scale copies.
//
// Roles (8 warps; 12 with the scale writers; 16 in the converting forms):
//   warp 0      TMA producer: per K stage (128 K, or 256 K for the fp4 kinds on chunkable
//               scale rows) the weight tile [128 x K] and the token tile [tn x K] into a
//               STAGES-deep ring: e4m3 (and padded e2m1) rows of 128 bytes per box, 128-byte
//               swizzle; packed e2m1 rows of 64 bytes (64-byte swizzle) or 128 bytes for the
//               fp4 kinds; packed rows of 64 bytes unswizzled for the converting forms.
//   warp 1      TMEM owner + MMA thread: per stage (without scale writers) tcgen05.cp of
//               both scale blocks into TMEM, then 4 x tcgen05.mma kind::mxf8f6f4.block_scale
//               per 128 K (K = 32 each, the scale-factor id picks the byte of the 4-byte
//               scale word; kind::mxf4 / kind::mxf4nvf4: 2 x K = 64; converted nvfp4: 8 x
//               kind::f16, K = 16), accumulating over all of K in a 2-deep TMEM
//               accumulator ring.
//   warps 2, 3  scale loaders (token rows, weight rows): per stage each row's 4 UE8M0 codes
//               (one 4-byte word, row-major source) are cp.async'ed into the packed
//               512-byte block (row r at byte (r%32)*16 + (r/32)*4); a few stages in
//               flight.  With pre-packed weight scales the producer copies the weight block
//               and warp 3 idles.  nvfp4: each row's 8 e4m3 codes of the stage, as two
//               packed blocks (codes 0-3 and 4-7) for the MMA kind, or row-major for the
//               converters.
//   warps 4-7   epilogue: warp w holds weight rows 32*(w%4).. of the tile, reads the tn
//               token columns of the accumulator, rounds to bf16 and stores C[m, n] for the
//               tile's token rows that belong to the expert.
//   warps 8-11  (fp4 kinds, and MXFP8 tiles of up to 64 token rows) scale writers: warp
//               8 + q stores TMEM lane quarter q of each
//               stage's scale slot with tcgen05.st (one slot per ring stage), so the MMA
//               thread issues only MMAs and the commit.  With chunkable scale rows (16
//               aligned bytes = 4 stages of UE8M0 or 2 of UE4M3 codes) each writer fetches its
//               own weight row's and all token rows' chunks, several groups ahead, into
//               private staging slots, and warps 2 and 3 idle; otherwise they relay the
//               loaders' packed blocks.
//   warps 8-15  (converting forms, tn <= 64) converters: each converted slot takes every
//               CSTAGES-th stage, whose packed weight tile (and packed token tile) its warp
//               (nvfp4: its two warps, half the rows each) re-encodes from the load ring into
//               the slot's e4m3 (fp16) tiles, which the MMA reads; the load ring
//               stays deep (up to 16 stages of 8 KB weight tiles) to keep HBM requests in
//               flight.  Warps 9 and 13 idle: they would share the MMA thread's
//               sub-partition, whose issue slots its tcgen05 instructions need.
#include <atomic>
#include <cuda_bf16.h>
#include "common.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace bsfp8 {
namespace mx {

constexpr int BK = 128;              // K per stage
constexpr int WROWS = 128;           // weight rows per tile (MMA M)
constexpr int EPI_WARP0 = 4;
constexpr int CONV_WARP0 = 8;        // converter warps 8..15 but 9, 13 (converting forms)
constexpr int SFW_WARP0 = 8;         // scale writer warps 8..11 (fp4 MMA kinds)

// Converter index of warp 8..15 (0..5), or -1 for warps 9 and 13 (sub-partition 1, the MMA
// thread's: its tcgen05 instructions need that sub-partition's issue slots).
__device__ __forceinline__ int converter_index(uint32_t warp) {
  const int w = (int)warp - CONV_WARP0;
  if (w < 0 || (w & 3) == 1) return -1;
  return (w >> 2) * 3 + ((w & 3) == 0 ? 0 : (w & 3) - 1);
}
constexpr uint32_t SMEM_LIMIT = 232448;  // dynamic shared memory per block (227 KB)

// Operand formats of a launch: A (tokens) x B (weights).
enum Format : int {
  FMT_MXFP8 = 0,        // e4m3 x e4m3
  FMT_MXFP8_MXFP4 = 1,  // e4m3 x e2m1
  FMT_MXFP4 = 2,        // e2m1 x e2m1
  FMT_NVFP4 = 3,        // e2m1 x e2m1 with e4m3 scales per 16 (fp16 MMA on dequantized tiles)
  FMT_MXFP4_MMA = 4,    // e2m1 x e2m1, kind::mxf4 on the packed tiles as loaded
  FMT_NVFP4_MMA = 5,    // e2m1 x e2m1 with UE4M3 scales per 16, kind::mxf4nvf4 (scale_vec::4X)
  FMT_MXFP8_MXFP4_MMA = 6,  // e4m3 x e2m1, kind::mxf8f6f4 on e2m1 weight tiles that TMA loads
                            // padded (16 codes in each 16 bytes' first 8)
};
constexpr int SF_BLOCK = 512;        // packed scale block: 128 rows x 4 codes
constexpr int SCALE_LOOKAHEAD = 4;   // scale stages in flight per loader warp
constexpr int STG_SLOTS = 3;         // staged 16-byte groups: one in use, two in flight
constexpr uint32_t STG_SLOT = WROWS * 16;

template <int TN_, int FMT_ = FMT_MXFP8, int SK_ = 128>
struct Cfg {
  static constexpr int TN = TN_;                               // token rows per tile
  static constexpr int FMT = FMT_;
  // fp4 MMA kinds: the packed tiles feed the tensor core as loaded (64-byte swizzle, K = 64
  // per MMA), no converter warps
  static constexpr bool NATIVE =
      FMT_ == FMT_MXFP4_MMA || FMT_ == FMT_NVFP4_MMA || FMT_ == FMT_MXFP8_MXFP4_MMA;
  // e4m3 tokens with e2m1 weights on kind::mxf8f6f4: the weight tile in shared memory has a
  // byte per element (the padded layout), K = 32 per MMA as for e4m3
  static constexpr bool MIXED = FMT_ == FMT_MXFP8_MXFP4_MMA;
  // K per stage: 128, or 256 for the fp4 kinds on chunkable scale rows (16 KB weight stages of
  // 128-byte rows, 128-byte swizzle, four K = 64 MMAs and one commit per stage)
  static constexpr int SK = SK_;
  static constexpr bool WIDE = SK_ == 256;
  static_assert(SK_ == 128 || (NATIVE && SK_ == 256), "256-K stages for the fp4 kinds only");
  static constexpr bool NV = FMT_ == FMT_NVFP4 || FMT_ == FMT_NVFP4_MMA;
  static constexpr bool B_FP4 = FMT_ != FMT_MXFP8;
  static constexpr bool A_FP4 = FMT_ != FMT_MXFP8 && FMT_ != FMT_MXFP8_MXFP4 && !MIXED;
  static constexpr bool CONVERT = B_FP4 && !NATIVE;
  static constexpr bool NV_F16 = NV && CONVERT;  // nvfp4 dequantized for the fp16 MMA
  // Scale feed: the MMA thread copies each stage's scale blocks into TMEM (tcgen05.cp), or
  // (SF_ST) four writer warps, one per TMEM lane quarter, store them (tcgen05.st) into a
  // per-stage TMEM slot and the MMA thread issues only MMAs and the commit.  128-row MXFP8
  // tiles keep the copies: the writers' token staging (every writer holds all token rows)
  // would cost a ring stage there.
  static constexpr bool SF_ST = NATIVE || (FMT_ == FMT_MXFP8 && TN_ <= 64);
  static constexpr int THREADS = CONVERT ? 512 : SF_ST ? 384 : 256;
  static_assert(!CONVERT || TN <= 64, "converting fp4 tiles hold at most 64 token rows");
  // bytes per converted element: e4m3 for the MX formats, fp16 for nvfp4
  static constexpr uint32_t ESZ = NV ? 2 : 1;
  // scale bytes per stage: packed UE8M0 blocks (MX), row-major e4m3 codes per 16 K (nvfp4 for
  // the fp16 MMA), or two packed UE4M3 blocks, one per K = 64 MMA (nvfp4 MMA kind)
  // 4-column TMEM scale groups per operand and stage: one per 128 K of UE8M0 codes, one per
  // K = 64 MMA of UE4M3 codes
  static constexpr int SF_GROUPS = !NATIVE ? 1 : NV ? SK / 64 : SK / 128;
  static_assert(!SF_ST || NATIVE || SK == 128, "e4m3 stages hold 128 K");
  // (wide stages: the scale writers fetch the codes themselves; the weight blocks stay for
  // pre-packed MX weight scales, which the producer copies with the stage)
  static constexpr uint32_t SFW_STAGE =
      NV_F16 ? WROWS * (BK / 16) : (WIDE && NV) ? 0 : SF_GROUPS * SF_BLOCK;
  static constexpr uint32_t SFT_STAGE = WIDE ? 0 : SF_GROUPS * SF_BLOCK;
  static_assert(!NV_F16 || TN * (BK / 16) <= SFT_STAGE, "nvfp4 token scales of a stage");
  // Load ring (STAGES deep): per stage the weight tile, the token tile and the scale
  // blocks as they arrive (the row layouts of the producer's comment at the top).  Offsets
  // of a stage along a row: W_KX, T_KX.
  static constexpr uint32_t W_STAGE = (B_FP4 && !MIXED) ? WROWS * SK / 2 : WROWS * SK;
  static constexpr uint32_t T_STAGE = A_FP4 ? TN * SK / 2 : TN * SK;
  // TMA x of a stage: bytes, or e2m1 elements for the padded weight map
  static constexpr int W_KX = (B_FP4 && !MIXED) ? SK / 2 : SK;
  static constexpr int T_KX = A_FP4 ? SK / 2 : SK;
  // TMA boxes per operand and stage: a box is 128 bytes (or 128 padded e2m1 elements) wide
  static constexpr int W_BOXES = MIXED ? SK / 128 : 1;
  static constexpr int T_BOXES = A_FP4 ? 1 : SK / 128;
  // Converted ring (fp4 formats): the e4m3 (fp16) tiles the MMA reads in place of the packed
  // ones; slot c takes the stages i with i % CSTAGES == c, converted by SPLIT warps that
  // share the rows of each stage (nvfp4's dequantization is the heavier, and its 40 KB
  // slots leave room for three).  The load ring keeps the HBM requests in flight.
  static constexpr int CSTAGES = !CONVERT ? 0 : NV ? 3 : (A_FP4 && TN > 32) ? 4 : 6;
  static constexpr int SPLIT = NV ? 2 : 1;
  static constexpr int NCONV = CSTAGES * SPLIT;  // converter warps (at most 6)
  static constexpr uint32_t CW_STAGE = CONVERT ? WROWS * BK * ESZ : 0;  // 16 KB (32 KB fp16)
  static constexpr uint32_t CT_STAGE = A_FP4 ? TN * BK * ESZ : 0;
  static constexpr uint32_t CONV_BYTES = CSTAGES * (CW_STAGE + CT_STAGE);
  static constexpr uint32_t PER_STAGE = W_STAGE + T_STAGE + SFW_STAGE + SFT_STAGE;
  // staged scale loads (both operands): STG_AHEAD groups of 16-byte row chunks in flight:
  // 8 stages ahead for e4m3 tiles; 1536 K (12 stages of 128 K, 6 of 256 K) for the fp4 kinds
  static constexpr int CPS = NV ? SK / 16 : SK / 32;  // scale codes per row and stage
  static constexpr int GS = 16 / CPS;                 // stages per 16-byte chunk
  // (128-row token tiles: at most 3 groups, each writer keeping 2 KB of token chunks per slot)
  static constexpr int STG_AHEAD_K = NATIVE ? (1536 / SK) / GS : STG_SLOTS - 1;
  static constexpr int STG_AHEAD = (TN >= 128 && STG_AHEAD_K > 3) ? 3 : STG_AHEAD_K;
  static constexpr int STG_N = STG_AHEAD + 1;
  // staging per slot: 128 weight rows and the token rows (x4 with the scale writers, each of
  // which keeps its own copy of the token rows)
  static constexpr uint32_t STGT_SLOT = (SF_ST ? 4 : 1) * TN * 16;
  static constexpr uint32_t STG_BYTES = STG_N * (STG_SLOT + STGT_SLOT);
  // fp4: as many load stages as fit next to the converted ring (if any), the staging slots,
  // the barriers and the alignment pad, at most 16 (128 KB of packed weights in flight)
  static constexpr int FIT =
      (int)((SMEM_LIMIT - CONV_BYTES - STG_BYTES - 2048) / PER_STAGE);
  // the scale writers' per-stage TMEM slots share the 512 columns with the accumulators
  static constexpr int TMEM_FIT = SF_ST ? (int)((512 - 2 * TN) / (8 * SF_GROUPS)) : 16;
  static constexpr int FIT_ALL = FIT < TMEM_FIT ? FIT : TMEM_FIT;
  static constexpr int STAGES = !B_FP4 ? ((TN <= 32) ? 10 : (TN <= 64) ? 8 : 6)
                                       : (FIT_ALL < 16 ? FIT_ALL : 16);
  static constexpr int LOOKAHEAD = SCALE_LOOKAHEAD < STAGES - 1 ? SCALE_LOOKAHEAD : STAGES - 1;
  // the epilogue's factor: 2^6 per fp4 operand undoes the re-encoding's 2^-6 (exact in fp32)
  static constexpr float POST = (NV || NATIVE) ? 1.0f : A_FP4 ? 4096.0f : (B_FP4 ? 64.0f : 1.0f);
  static constexpr uint32_t SMEM_CW = 0;
  static constexpr uint32_t SMEM_CT = SMEM_CW + CSTAGES * CW_STAGE;
  static constexpr uint32_t SMEM_W = SMEM_CT + CSTAGES * CT_STAGE;
  static constexpr uint32_t SMEM_T = SMEM_W + STAGES * W_STAGE;
  static constexpr uint32_t SMEM_SFW = SMEM_T + STAGES * T_STAGE;
  static constexpr uint32_t SMEM_SFT = SMEM_SFW + STAGES * SFW_STAGE;
  // weight-scale staging of the grouped loader: STG_N x (128 rows x 16 bytes), STG_AHEAD
  // groups in flight
  static constexpr uint32_t SMEM_STG = SMEM_SFT + STAGES * SFT_STAGE;
  static constexpr uint32_t SMEM_STGT = SMEM_STG + STG_N * STG_SLOT;  // token staging
  static constexpr uint32_t SMEM_CTL = SMEM_STGT + STG_N * STGT_SLOT;
  // bytes a stage's loads complete on its barrier (the padded e2m1 weight load counts the
  // packed bytes it reads, half the shared-memory tile)
  static constexpr uint32_t STAGE_TX = (MIXED ? W_STAGE / 2 : W_STAGE) + T_STAGE;
  // TMEM: 2 accumulators of TN columns, then 2 slots each of weight / token scales (4 columns
  // per scale group, every group on a 4-column boundary)
  static constexpr uint32_t ACC_COLS = 2 * TN;
  static constexpr uint32_t SF_COLS = 4 * SF_GROUPS;  // columns of one slot
  static constexpr uint32_t SFW_COL = ACC_COLS;
  static constexpr uint32_t SFT_COL = ACC_COLS + 2 * SF_COLS;
  // SF_ST: one slot pair per operand-ring stage (weights, then tokens)
  static constexpr uint32_t SF_STAGE_COLS = 2 * SF_COLS;
  static constexpr uint32_t TMEM_USED =
      SF_ST ? ACC_COLS + STAGES * SF_STAGE_COLS : ACC_COLS + 4 * SF_COLS;
  static constexpr uint32_t TMEM_COLS = (TMEM_USED <= 64) ? 64 : (TMEM_USED <= 128) ? 128
                                        : (TMEM_USED <= 256) ? 256 : 512;
  static_assert(TMEM_USED <= 512, "accumulators and scale slots fit the 512 TMEM columns");
  static_assert(LOOKAHEAD >= 1 && LOOKAHEAD < STAGES, "scale look-ahead must leave a free stage");
  static_assert(STAGES > CSTAGES, "the load ring is deeper than the converted ring");
  // 128-byte-swizzled tiles start on 1024-byte boundaries
  static_assert(SMEM_W % 1024 == 0 && SMEM_T % 1024 == 0 && CT_STAGE % 1024 == 0, "swizzle");
  static_assert(A_FP4 || T_STAGE % 1024 == 0, "token tiles keep the 1024-byte alignment");
  // 64-byte-swizzled packed tiles (fp4 MMA kinds) start on 512-byte boundaries, 128-byte-
  // swizzled ones (wide stages) on 1024-byte boundaries
  static_assert(!NATIVE || (W_STAGE % 512 == 0 && T_STAGE % 512 == 0), "64-byte swizzle");
  static_assert(!WIDE || (W_STAGE % 1024 == 0 && T_STAGE % 1024 == 0), "128-byte swizzle");
  static_assert(!NATIVE || CPS * GS == 16, "a 16-byte chunk holds whole stages of codes");
  static_assert(B_FP4 || W_STAGE % 1024 == 0, "weight tiles keep the 1024-byte alignment");
};

template <class C>
struct Ctl {
  uint64_t full[C::STAGES];
  uint64_t empty[C::STAGES];
  uint64_t cfull[C::CSTAGES > 0 ? C::CSTAGES : 1];  // converted tiles written (fp4 formats)
  uint64_t sfull[C::SF_ST ? C::STAGES : 1];          // stage's scales stored in TMEM (SF_ST)
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  int valid;
  int pad;
  long long total_tiles;
};

template <class C>
constexpr uint32_t smem_bytes() {
  return C::SMEM_CTL + sizeof(Ctl<C>) + 1024;
}

// Four e2m1 pairs (one 32-bit word of a packed row: element 2i in the low nibble of byte
// i) to eight e4m3 codes, each exactly 2^-6 times the e2m1 value: the sign moves from bit
// 3 of the nibble to bit 7 of the byte, the 3 magnitude bits to bits 2..4.
__device__ __forceinline__ uint2 e2m1x8_to_e4m3x8(uint32_t w) {
  const uint32_t lo = ((w << 4) & 0x80808080u) | ((w << 2) & 0x1C1C1C1Cu);  // even elements
  const uint32_t hi = (w & 0x80808080u) | ((w >> 2) & 0x1C1C1C1Cu);         // odd elements
  return make_uint2(__byte_perm(lo, hi, 0x5140), __byte_perm(lo, hi, 0x7362));
}

// Re-encode a packed tile [ROWS x 64 B] (128 e2m1 per row, row-major) into the e4m3 tile
// [ROWS x 128 B] with the 128-byte swizzle (16-byte chunk c of row r at chunk c ^ (r % 8)),
// one warp.  For a group of 8 rows, lane l reads 16 packed bytes (row l / 4 of the group,
// chunk l % 4: 32 elements) and writes output chunks 2*(l%4) and 2*(l%4)+1; eight
// consecutive lanes read 128 contiguous bytes and write 8 distinct chunks of two rows.  Four
// groups' loads are issued before their conversions.
template <int ROWS>
__device__ __forceinline__ void convert_fp4_tile(const uint8_t* raw, uint8_t* out,
                                                 uint32_t lane) {
  static_assert(ROWS % 32 == 0, "groups of 4 x 8 rows");
  const uint32_t q = lane & 3;
#pragma unroll 1
  for (int g0 = 0; g0 < ROWS / 8; g0 += 4) {
    uint4 in[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t row = (g0 + u) * 8 + (lane >> 2);
      in[u] = *reinterpret_cast<const uint4*>(raw + row * 64 + q * 16);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t row = (g0 + u) * 8 + (lane >> 2);
      const uint2 a = e2m1x8_to_e4m3x8(in[u].x), b = e2m1x8_to_e4m3x8(in[u].y);
      const uint2 c = e2m1x8_to_e4m3x8(in[u].z), d = e2m1x8_to_e4m3x8(in[u].w);
      uint8_t* orow = out + row * 128;
      *reinterpret_cast<uint4*>(orow + (((2 * q) ^ (row & 7)) << 4)) =
          make_uint4(a.x, a.y, b.x, b.y);
      *reinterpret_cast<uint4*>(orow + (((2 * q + 1) ^ (row & 7)) << 4)) =
          make_uint4(c.x, c.y, d.x, d.y);
    }
  }
}

// Eight e2m1 (one 32-bit word of a packed row, element 2i in the low nibble of byte i) times
// one fp16 scale (replicated in both halves of s): four fp16 pairs, lower element in the
// lower half.  Both conversions are exact, and so is the product: an e2m1 value has at most
// 2 significant bits and an e4m3 scale 4, and |value * scale| lies in [2^-10, 2688], inside
// the normal fp16 range.
__device__ __forceinline__ uint4 e2m1x8_scaled_f16x8(uint32_t w, uint32_t s) {
  uint4 o;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t"
      "mul.rn.f16x2 %0, %0, %5;\n\t"
      "mul.rn.f16x2 %1, %1, %5;\n\t"
      "mul.rn.f16x2 %2, %2, %5;\n\t"
      "mul.rn.f16x2 %3, %3, %5;\n\t}"
      : "=r"(o.x), "=r"(o.y), "=r"(o.z), "=r"(o.w)
      : "r"(w), "r"(s));
  return o;
}

// Two e4m3 scale codes (low byte first) to an fp16 pair, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t codes16) {
  uint32_t h;
  asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
      : "=r"(h)
      : "r"(codes16));
  return h;
}

// Dequantize a packed nvfp4 tile [ROWS x 64 B] with its e4m3 scales [ROWS x 8] (one per 16
// elements) into the fp16 tile the kind::f16 MMA reads: K-major, 128-byte swizzle, two
// atoms of 64 elements ([atom][ROWS][128 B], 16-byte chunk c of row r at c ^ (r % 8)).  One
// warp converts rows row0 .. row0 + PART - 1.  For a group of 8 rows lane l takes row l / 4,
// packed chunk q = l % 4 (elements 32q .. 32q+31, scale groups 2q and 2q+1) and writes its
// 64 output bytes as chunks 4*(q%2) .. 4*(q%2)+3 of atom q / 2; lanes of atom 1 store their
// chunks in the order 2, 3, 0, 1, so that each store of a quarter-warp covers 8 distinct
// chunk positions (32 banks) rather than 4 positions twice.
template <int ROWS, int PART>
__device__ __forceinline__ void convert_nvfp4_tile(const uint8_t* raw, const uint8_t* sc,
                                                   uint8_t* out, uint32_t lane, int row0) {
  static_assert(PART % 16 == 0 && ROWS % PART == 0, "groups of 2 x 8 rows");
  const uint32_t q = lane & 3;
  const bool second = (q >> 1) != 0;
  uint8_t* atom = out + (q >> 1) * (ROWS * 128);
#pragma unroll 1
  for (int g0 = row0 / 8; g0 < (row0 + PART) / 8; g0 += 2) {
    uint4 in[2];
    uint32_t s2[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t row = (g0 + u) * 8 + (lane >> 2);
      in[u] = *reinterpret_cast<const uint4*>(raw + row * 64 + q * 16);
      s2[u] = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sc + row * 8 + 2 * q));
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t row = (g0 + u) * 8 + (lane >> 2);
      const uint32_t s_lo = __byte_perm(s2[u], 0, 0x1010);  // scale of elements 0..15
      const uint32_t s_hi = __byte_perm(s2[u], 0, 0x3232);  // scale of elements 16..31
      uint4 o0 = e2m1x8_scaled_f16x8(in[u].x, s_lo);
      uint4 o1 = e2m1x8_scaled_f16x8(in[u].y, s_lo);
      uint4 o2 = e2m1x8_scaled_f16x8(in[u].z, s_hi);
      uint4 o3 = e2m1x8_scaled_f16x8(in[u].w, s_hi);
      uint32_t c0 = 4 * (q & 1), c1 = c0 + 1, c2 = c0 + 2, c3 = c0 + 3;
      if (second) {  // store order 2, 3, 0, 1
        const uint4 t0 = o0, t1 = o1;
        o0 = o2; o1 = o3; o2 = t0; o3 = t1;
        const uint32_t d0 = c0, d1 = c1;
        c0 = c2; c1 = c3; c2 = d0; c3 = d1;
      }
      const uint32_t r7 = row & 7;
      uint8_t* orow = atom + row * 128;
      *reinterpret_cast<uint4*>(orow + ((c0 ^ r7) << 4)) = o0;
      *reinterpret_cast<uint4*>(orow + ((c1 ^ r7) << 4)) = o1;
      *reinterpret_cast<uint4*>(orow + ((c2 ^ r7) << 4)) = o2;
      *reinterpret_cast<uint4*>(orow + ((c3 ^ r7) << 4)) = o3;
    }
  }
}

// Waits of every role but the MMA thread sleep in the barrier (mbar_wait_sleep): polling
// warps would take issue slots from the warps they share a sub-partition with (the MMA
// thread, the fp4 converters).  BSMX_SPIN_WAITS restores polling for comparison.
__device__ __forceinline__ bool role_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
#ifdef BSMX_SPIN_WAITS
  return mbar_wait(bar, parity, abort);
#else
  return mbar_wait_sleep(bar, parity, abort);
#endif
}

// The MMA thread polls: it alone issues the tensor-core work and must see each stage at once.
__device__ __forceinline__ bool mma_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
#ifdef BSMX_MMA_SLEEP
  return mbar_wait_sleep(bar, parity, abort);
#else
  return mbar_wait(bar, parity, abort);
#endif
}

__device__ __forceinline__ void record_error(int* err, int code, volatile int* abort) {
  atomicCAS(err, 0, code);
  *abort = 1;
}

// Descriptor of a packed 512-byte scale block for tcgen05.cp (32 rows x 16 bytes, no
// swizzle: 8-row core matrices of 128 bytes, 128 bytes apart).
__device__ __forceinline__ uint64_t sf_block_desc(uint32_t saddr) {
  return make_smem_desc(saddr, 0, 128, LAYOUT_NONE);
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
bsmxfp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const GemmArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Ctl<C>* ctl = reinterpret_cast<Ctl<C>*>(smem + C::SMEM_CTL);
  volatile int* abort = &ctl->abort;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const int KB = args.K / C::SK;  // stages per tile
  // bytes per row of a row-major scale matrix: UE8M0 per 32 K, or e4m3 per 16 K (nvfp4)
  const int scale_row = args.K / (C::NV ? 16 : 32);
  const bool packed_b = args.b_scales_packed != 0;
  // Scale writers fetching their own scale chunks (SF_ST, chunkable rows: each row's codes of
  // 16 / CPS consecutive stages form one aligned 16-byte chunk); otherwise the loader warps
  // pack each stage's blocks in shared memory and the writers relay them into TMEM.
  constexpr int CPS = C::NATIVE ? C::CPS : C::NV ? 8 : 4;  // scale codes per row per stage
  constexpr int GS = 16 / CPS;                               // stages per 16-byte chunk
  const bool sf_direct =
      C::SF_ST && KB % GS == 0 && scale_row % 16 == 0 &&
      reinterpret_cast<uintptr_t>(args.a_scales) % 16 == 0 &&
      (packed_b || reinterpret_cast<uintptr_t>(args.b_scales) % 16 == 0);
  // pre-packed weight-scale bytes per stage (one 512-byte block per 128 K)
  constexpr uint32_t PB_BYTES = (C::SK / 128) * SF_BLOCK;
  // Wide stages run with fetching writers only (the host launches them on chunkable rows):
  // anything else winds down before any barrier is used, with the error recorded.
  if (C::WIDE && !sf_direct) {
    if (threadIdx.x == 0) atomicCAS(args.err, 0, DEV_TIMEOUT);
    return;
  }

  // Tiles: per expert ceil(M_e / TN) token tiles x N/128 weight tiles (weights fastest).
  if (warp == 0) {
    int status;
    int64_t row_tiles;
    validate_offsets<C::TN>(args.offsets, args.expert_ids, args.E, args.num_experts, args.M_total,
                            args.min_group_rows, args.max_group_rows, DEV_BAD_OFFSETS, DEV_BAD_EXPERT_IDS, status, row_tiles);
    if (lane == 0) {
      ctl->valid = status == 0;
      ctl->total_tiles = row_tiles * (args.N / WROWS);
      ctl->abort = 0;
      if (status && blockIdx.x == 0) atomicCAS(args.err, 0, status);
    }
  }
  __syncthreads();
  const int64_t total_tiles = ctl->total_tiles;
  if (!ctl->valid || (int64_t)blockIdx.x >= total_tiles) return;

  const uint32_t sW = smem_u32(smem + C::SMEM_W);
  const uint32_t sT = smem_u32(smem + C::SMEM_T);
  const uint32_t sSFW = smem_u32(smem + C::SMEM_SFW);
  const uint32_t sSFT = smem_u32(smem + C::SMEM_SFT);
  auto full_bar = [&](int s) { return smem_u32(&ctl->full[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&ctl->empty[s]); };
  auto tfull_bar = [&](int s) { return smem_u32(&ctl->tfull[s]); };
  auto tempty_bar = [&](int s) { return smem_u32(&ctl->tempty[s]); };
  auto cfull_bar = [&](int s) { return smem_u32(&ctl->cfull[s]); };
  auto sfull_bar = [&](int s) { return smem_u32(&ctl->sfull[s]); };

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    for (int s = 0; s < C::STAGES; ++s) {
      // producer (with bytes) + token-scale loader (+ weight-scale loader)
      mbar_init(full_bar(s), sf_direct ? 1 : packed_b ? 2 : 3);
      mbar_init(empty_bar(s), 1);  // one MMA commit
    }
    for (int s = 0; s < C::CSTAGES; ++s) mbar_init(cfull_bar(s), C::SPLIT);  // its converters
    if constexpr (C::SF_ST)
      for (int s = 0; s < C::STAGES; ++s) mbar_init(sfull_bar(s), 4);  // the 4 scale writers
    for (int s = 0; s < 2; ++s) {
      mbar_init(tfull_bar(s), 1);
      mbar_init(tempty_bar(s), 4);  // the 4 epilogue warps
    }
    mbar_init(smem_u32(&ctl->mma_done), 1);
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc<1>(smem_u32(&ctl->tmem_base), C::TMEM_COLS);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    // =============================== TMA producer ===============================
    if (lane == 0) {
      GroupedScheduler<C::TN, WROWS> sched;
      const uint64_t pol_w = l2_policy_evict_first();  // weights stream once per token tile
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      bool ok = true;
      TileCoord tc;
      for (int64_t t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
        if (!sched.locate(args, t, tc)) break;
        const int32_t w_row = tc.be * args.N + tc.n0;
        const int32_t t_row = (int32_t)tc.m0;
        // packed weight scales: this tile's 128 rows, K block 0 (blocks of a row are adjacent,
        // one per 128 K)
        const uint8_t* w_sf = static_cast<const uint8_t*>(args.b_scales) +
                              ((int64_t)w_row / WROWS) * (args.K / 128) * SF_BLOCK;
        for (int kb = 0; kb < KB; ++kb) {
          if (!role_wait(empty_bar(stage), phase ^ 1, abort)) {
            record_error(args.err, DEV_TIMEOUT, abort);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), C::STAGE_TX + (packed_b ? PB_BYTES : 0u));
#pragma unroll
          for (int h = 0; h < C::W_BOXES; ++h)  // 128-element boxes into 128-row sub-tiles
            tma_load_2d_hint(sW + stage * C::W_STAGE + h * (WROWS * 128), &tmB,
                             kb * C::W_KX + h * 128, w_row, full_bar(stage), pol_w);
#pragma unroll
          for (int h = 0; h < C::T_BOXES; ++h)
            tma_load_2d(sT + stage * C::T_STAGE + h * (C::TN * 128), &tmA, kb * C::T_KX + h * 128,
                        t_row, full_bar(stage));
          if (packed_b)  // the stage's weight-scale block is stored ready-made
            bulk_copy_g2s_hint(sSFW + stage * C::SFW_STAGE, w_sf + (int64_t)kb * PB_BYTES,
                               PB_BYTES, full_bar(stage), pol_w);
          ++issued;
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
      }
      // The last loads have landed before the CTA can exit: once the MMA consumed a stage
      // it had landed; wait (bounded) for the stages the MMA did not get to.
      const int64_t pending = issued < C::STAGES ? issued : C::STAGES;
      for (int64_t i = 0; i < pending; ++i) {
        stage = (stage + C::STAGES - 1) % C::STAGES;
        if (stage == C::STAGES - 1) phase ^= 1;
        mbar_wait_timed(empty_bar(stage), phase);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================ MMA thread ================================
    if (lane == 0) {
      GroupedScheduler<C::TN, WROWS> sched;
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0, slot = 0;
      uint32_t cstage = 0, cphase = 0;  // converted ring (fp4 formats)
      bool ok = true;
      TileCoord tc;
      for (int64_t t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
        if (!sched.locate(args, t, tc)) break;
        if (!mma_wait(tempty_bar(acc), acc_phase ^ 1, abort)) {
          record_error(args.err, DEV_TIMEOUT, abort);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * C::TN;
        for (int kb = 0; kb < KB; ++kb) {
          // fp4: the converters have written this stage's e4m3 tiles (after its loads and
          // scale blocks landed); otherwise the stage's loads themselves
          const bool got = C::CONVERT ? mma_wait(cfull_bar(cstage), cphase, abort)
                           : C::SF_ST ? mma_wait(sfull_bar(stage), phase, abort)
                                      : mma_wait(full_bar(stage), phase, abort);
          if (!got) {
            record_error(args.err, DEV_TIMEOUT, abort);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfw_t = C::SF_ST ? tmem_base + C::ACC_COLS + stage * C::SF_STAGE_COLS
                                          : tmem_base + C::SFW_COL + C::SF_COLS * slot;
          const uint32_t sft_t = C::SF_ST ? sfw_t + C::SF_COLS
                                          : tmem_base + C::SFT_COL + C::SF_COLS * slot;
          if constexpr (!C::NV_F16 && !C::SF_ST) {
#pragma unroll
            for (int g = 0; g < C::SF_GROUPS; ++g) {
              tmem_cp_32x128b_warpx4<1>(sfw_t + 4 * g,
                                        sf_block_desc(sSFW + stage * C::SFW_STAGE + g * SF_BLOCK));
              tmem_cp_32x128b_warpx4<1>(sft_t + 4 * g,
                                        sf_block_desc(sSFT + stage * C::SFT_STAGE + g * SF_BLOCK));
            }
          }
          const uint32_t w_tile = C::CONVERT ? smem_u32(smem + C::SMEM_CW) + cstage * C::CW_STAGE
                                             : sW + stage * C::W_STAGE;
          const uint32_t t_tile = C::A_FP4 ? smem_u32(smem + C::SMEM_CT) + cstage * C::CT_STAGE
                                           : sT + stage * C::T_STAGE;
          const uint64_t wdesc = kmajor_sw128_desc(w_tile);
          const uint64_t tdesc = kmajor_sw128_desc(t_tile);
          if constexpr (C::CONVERT) {
            if (++cstage == C::CSTAGES) { cstage = 0; cphase ^= 1; }
          }
          if constexpr (C::MIXED) {
            // e2m1 weights (padded: a byte per element, 128-byte rows, 128-byte swizzle) and
            // e4m3 tokens, in 128-K sub-tiles: K = 32 per MMA, the scale-factor id picks the
            // byte of the sub-tile's scale word
#pragma unroll
            for (int k = 0; k < C::SK / 32; ++k) {
              const int sub = k >> 2, kk = k & 3;
              umma_mxf8f6f4<1>(d_tmem, wdesc + (uint64_t)((sub * WROWS * 128) >> 4) + kk * 2,
                               tdesc + (uint64_t)((sub * C::TN * 128) >> 4) + kk * 2,
                               idesc_mxf8f6f4(WROWS, C::TN, MXF_E2M1, MXF_E4M3, kk, kk),
                               sfw_t + 4 * sub, sft_t + 4 * sub, (kb > 0 || k > 0) ? 1u : 0u);
            }
          } else if constexpr (C::NATIVE) {
            // packed e2m1 tiles of 64-byte rows (64-byte swizzle) or 128-byte rows (wide
            // stages, 128-byte swizzle): a K = 64 MMA every 32 bytes
            const uint64_t wd = C::WIDE ? kmajor_sw128_desc(sW + stage * C::W_STAGE)
                                        : kmajor_sw64_desc(sW + stage * C::W_STAGE);
            const uint64_t td = C::WIDE ? kmajor_sw128_desc(sT + stage * C::T_STAGE)
                                        : kmajor_sw64_desc(sT + stage * C::T_STAGE);
#pragma unroll
            for (int k = 0; k < C::SK / 64; ++k) {
              if constexpr (C::NV)  // UE4M3 per 16: the k-th scale group of each operand
                umma_mxf4nvf4_4x(d_tmem, wd + (uint64_t)(k * 2), td + (uint64_t)(k * 2),
                                 idesc_nvf4_e2m1_ue4m3(WROWS, C::TN), sfw_t + 4 * k, sft_t + 4 * k,
                                 (kb > 0 || k > 0) ? 1u : 0u);
              else  // UE8M0 per 32: group k / 2, bytes 2 (k % 2), +1 of its scale word
                umma_mxf4(d_tmem, wd + (uint64_t)(k * 2), td + (uint64_t)(k * 2),
                          idesc_mxf4_e2m1(WROWS, C::TN, 2 * (k & 1), 2 * (k & 1)),
                          sfw_t + 4 * (k >> 1), sft_t + 4 * (k >> 1),
                          (kb > 0 || k > 0) ? 1u : 0u);
            }
          } else if constexpr (C::NV_F16) {
            // fp16 tiles: two 64-element swizzle atoms per stage, K = 16 per MMA
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              const uint64_t wd = kmajor_sw128_desc(w_tile + (k >> 2) * (WROWS * 128)) +
                                  (uint64_t)((k & 3) * 2);
              const uint64_t td = kmajor_sw128_desc(t_tile + (k >> 2) * (C::TN * 128)) +
                                  (uint64_t)((k & 3) * 2);
              umma_f16<1>(d_tmem, wd, td, idesc_f16_f32(WROWS, C::TN), (kb > 0 || k > 0) ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int k = 0; k < BK / 32; ++k)
              umma_mxf8f6f4<1>(d_tmem, wdesc + (uint64_t)(k * 2), tdesc + (uint64_t)(k * 2),
                               idesc_mxf8f6f4_e4m3(WROWS, C::TN, k, k), sfw_t, sft_t,
                               (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(empty_bar(stage));
          slot ^= 1;
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
      // every MMA issued has finished before TMEM is released; a wait that gives up is
      // reported and waited out once more (bounded) before the teardown
      umma_commit(smem_u32(&ctl->mma_done));
      if (!mbar_wait_timed(smem_u32(&ctl->mma_done), 0)) {
        record_error(args.err, DEV_TIMEOUT, abort);
        mbar_wait_timed(smem_u32(&ctl->mma_done), 0);
      }
    }
    __syncwarp();
  } else if (!C::WIDE && !sf_direct && (warp == 2 || (warp == 3 && !packed_b))) {
    // =============================== scale loaders ===============================
    // Warp 2 gathers the token rows' scales, warp 3 the weight rows' (unless they arrive
    // pre-packed with the producer's copies), into each stage's packed block(s): row r's 4
    // codes at byte (r % 32) * 16 + (r / 32) * 4.  Staged (below) when the rows' codes come
    // in aligned 16-byte chunks; otherwise each lane cp.async's 4-byte words (8 bytes per row
    // for the fp16 nvfp4 form) into the stage once its ring slot is free, and a stage is
    // announced on its full barrier once its copies have landed, C::LOOKAHEAD stages
    // (SCALE_LOOKAHEAD, fewer in a short ring) behind the newest issued one; token rows >= TN
    // of every block stay zero (written once here).
    const bool weights = warp == 3;
    const uint8_t* a_sc = static_cast<const uint8_t*>(args.a_scales);
    const uint8_t* b_sc = static_cast<const uint8_t*>(args.b_scales);
    if (!C::NV_F16 && !weights && C::TN < WROWS) {
      for (int s = 0; s < C::STAGES * C::SF_GROUPS; ++s)
        for (int rg = C::TN / 32; rg < 4; ++rg)
          *reinterpret_cast<uint32_t*>(smem + C::SMEM_SFT + s * SF_BLOCK + lane * 16 + rg * 4) = 0u;
    }
    GroupedScheduler<C::TN, WROWS> sched;
    uint32_t stage = 0, phase = 0;
    uint32_t ring[C::LOOKAHEAD + 1] = {};
    int inflight = 0, head = 0;
    bool ok = true;
    TileCoord tc;
    auto announce_oldest = [&]() {
      fence_proxy_async_smem();  // generic-proxy writes -> tcgen05.cp (async proxy)
      __syncwarp();
      if (lane == 0) mbar_arrive(full_bar(ring[head]));
      head = (head + 1) % (C::LOOKAHEAD + 1);
      --inflight;
    };
    // Staged: when a row's codes for GS consecutive stages form one aligned 16-byte chunk
    // (4 stages of 4 UE8M0 codes, or 2 stages of 8 UE4M3 codes), fetch each row's chunk with
    // one 16-byte copy STG_AHEAD groups ahead into a staging slot, and when a stage's ring
    // slot is free transpose its words into the stage's packed block(s): the DRAM latency of
    // the scales is covered by the staging slots, not by the ring.  Token rows past M_total
    // read as zero; rows >= TN of a token block are written zero.
    const uint8_t* sc_base = weights ? b_sc : a_sc;
    const bool grouped = !C::NV_F16 && (KB % GS == 0) && (scale_row % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(sc_base) % 16 == 0);
    if (grouped) {
      const int G = KB / GS;
      const int R = weights ? WROWS : C::TN;  // rows of the operand tile
      const uint32_t slot_bytes = (uint32_t)R * 16;
      const uint32_t sSTG = smem_u32(smem + (weights ? C::SMEM_STG : C::SMEM_STGT));
      const uint8_t* stg = smem + (weights ? C::SMEM_STG : C::SMEM_STGT);
      const uint32_t blk0 = weights ? C::SMEM_SFW : C::SMEM_SFT;
      const uint32_t blk_stage = weights ? C::SFW_STAGE : C::SFT_STAGE;
      GroupedScheduler<C::TN, WROWS> pre;
      TileCoord tp;
      int64_t tp_t = blockIdx.x;
      bool pre_ok = pre.locate(args, tp_t, tp);
      int qp = 0;
      auto issue_group = [&](int slot) {
        if (pre_ok) {
#pragma unroll
          for (int jr = 0; jr < 4; ++jr) {
            const int r = 32 * jr + (int)lane;
            if (r < R) {
              const uint8_t* src;
              uint32_t n = 16u;
              if (weights) {
                src = b_sc + ((int64_t)tp.be * args.N + tp.n0 + r) * scale_row + 16 * qp;
              } else {
                const int64_t m = tp.m0 + r;
                n = m < args.M_total ? 16u : 0u;
                src = n ? a_sc + m * scale_row + 16 * qp : a_sc;
              }
              cp_async_16(sSTG + slot * slot_bytes + r * 16, src, n);
            }
          }
          if (++qp == G) {
            qp = 0;
            tp_t += gridDim.x;
            pre_ok = tp_t < total_tiles && pre.locate(args, tp_t, tp);
          }
        }
        cp_async_commit();  // an empty group keeps the group count in step
      };
      for (int a = 0; a < C::STG_AHEAD; ++a) issue_group(a);
      int64_t g = 0;
      for (int64_t t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
        if (!sched.locate(args, t, tc)) break;
        for (int q = 0; ok && q < G; ++q, ++g) {
          cp_async_wait_group<C::STG_AHEAD - 1>();  // group g has landed (later ones in flight)
          __syncwarp();
          const uint8_t* src = stg + (g % C::STG_N) * slot_bytes;
          for (int j = 0; j < GS; ++j) {
            const bool got =
                __all_sync(0xffffffffu, role_wait(empty_bar(stage), phase ^ 1, abort));
            if (!got) {
              if (lane == 0) record_error(args.err, DEV_TIMEOUT, abort);
              ok = false;
              break;
            }
            // packed block b (the stage's codes 4b..4b+3): row 32*rg + lane at byte
            // lane*16 + rg*4
#pragma unroll
            for (int b = 0; b < CPS / 4; ++b) {
              uint32_t w[4];
#pragma unroll
              for (int rg = 0; rg < 4; ++rg)
                w[rg] = 32 * rg < R ? *reinterpret_cast<const uint32_t*>(
                                          src + (32 * rg + lane) * 16 + CPS * j + 4 * b)
                                    : 0u;
              *reinterpret_cast<uint4*>(smem + blk0 + stage * blk_stage + b * SF_BLOCK +
                                        lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            fence_proxy_async_smem();  // generic-proxy writes -> tcgen05.cp (async proxy)
            __syncwarp();
            if (lane == 0) mbar_arrive(full_bar(stage));
            if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          __syncwarp();
          issue_group((int)((g + C::STG_AHEAD) % C::STG_N));  // the slot group g - 1 used is free
        }
      }
      cp_async_wait_group<0>();
    }
    for (int64_t t = blockIdx.x; !grouped && ok && t < total_tiles; t += gridDim.x) {
      if (!sched.locate(args, t, tc)) break;
      const uint8_t* w_rows = b_sc + ((int64_t)tc.be * args.N + tc.n0) * scale_row;
      for (int kb = 0; kb < KB; ++kb) {
        const bool got = __all_sync(0xffffffffu, role_wait(empty_bar(stage), phase ^ 1, abort));
        if (!got) {
          if (lane == 0) record_error(args.err, DEV_TIMEOUT, abort);
          ok = false;
          break;
        }
        if (C::NV && C::NATIVE) {
          // nvfp4, MMA kind: row r's 8 UE4M3 codes of the stage, codes 0-3 (the first K = 64
          // MMA) into block 0 and codes 4-7 into block 1, each at byte (r % 32) * 16 + (r / 32) * 4
          const uint32_t d =
              (weights ? sSFW + stage * C::SFW_STAGE : sSFT + stage * C::SFT_STAGE) + lane * 16;
          if (weights) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint8_t* src = w_rows + (int64_t)(j * 32 + (int)lane) * scale_row + 8 * kb;
              cp_async_4(d + 4 * j, src, 4);
              cp_async_4(d + SF_BLOCK + 4 * j, src + 4, 4);
            }
          } else {
#pragma unroll
            for (int j = 0; j < C::TN / 32; ++j) {
              const int64_t m = tc.m0 + j * 32 + (int)lane;
              const bool live = m < args.M_total;
              const uint8_t* src = live ? a_sc + m * scale_row + 8 * kb : a_sc;
              cp_async_4(d + 4 * j, src, live ? 4u : 0u);
              cp_async_4(d + SF_BLOCK + 4 * j, live ? src + 4 : a_sc, live ? 4u : 0u);
            }
          }
        } else if (C::NV) {
          // nvfp4: row r's 8 e4m3 codes of the stage to byte 8r (row-major, as stored)
          const uint32_t d = weights ? sSFW + stage * C::SFW_STAGE : sSFT + stage * C::SFT_STAGE;
          const int rows = weights ? WROWS : C::TN;
#pragma unroll
          for (int j = 0; j < WROWS / 32; ++j) {
            const int r = j * 32 + (int)lane;
            if (r < rows) {
              if (weights) {
                cp_async_8(d + 8 * r, w_rows + (int64_t)r * scale_row + 8 * kb, 8);
              } else {
                const int64_t m = tc.m0 + r;
                const bool live = m < args.M_total;
                cp_async_8(d + 8 * r, live ? a_sc + m * scale_row + 8 * kb : a_sc, live ? 8u : 0u);
              }
            }
          }
        } else if (weights) {
          const uint32_t dw = sSFW + stage * C::SFW_STAGE + lane * 16;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = j * 32 + (int)lane;
            cp_async_4(dw + 4 * j, w_rows + (int64_t)r * scale_row + 4 * kb, 4);
          }
        } else {
          const uint32_t dt = sSFT + stage * C::SFT_STAGE + lane * 16;
#pragma unroll
          for (int j = 0; j < C::TN / 32; ++j) {
            const int64_t m = tc.m0 + j * 32 + (int)lane;
            const bool live = m < args.M_total;
            cp_async_4(dt + 4 * j, live ? a_sc + m * scale_row + 4 * kb : a_sc, live ? 4u : 0u);
          }
        }
        cp_async_commit();
        ring[(head + inflight) % (C::LOOKAHEAD + 1)] = stage;
        ++inflight;
        if (inflight > C::LOOKAHEAD) {
          cp_async_wait_group<C::LOOKAHEAD>();
          announce_oldest();
        }
        if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
      }
    }
    cp_async_wait_group<0>();
    while (inflight > 0) announce_oldest();
  } else if (warp >= EPI_WARP0 && warp < EPI_WARP0 + 4) {
    // ================================= epilogue =================================
    const uint32_t quarter = warp & 3;
    __nv_bfloat16* Cmat = static_cast<__nv_bfloat16*>(args.C);
    GroupedScheduler<C::TN, WROWS> sched;
    uint32_t acc = 0, acc_phase = 0;
    TileCoord tc;
    for (int64_t t = blockIdx.x; t < total_tiles; t += gridDim.x) {
      if (!sched.locate(args, t, tc)) break;
      const bool got = __all_sync(0xffffffffu, role_wait(tfull_bar(acc), acc_phase, abort));
      if (!got) {
        if (lane == 0) record_error(args.err, DEV_TIMEOUT, abort);
        break;
      }
      tc_fence_after();
      const int n = tc.n0 + (int)(quarter * 32 + lane);
      const uint32_t taddr = tmem_base + ((quarter * 32) << 16) + acc * C::TN;
      uint32_t v[C::TN];
#pragma unroll
      for (int c = 0; c < C::TN / 32; ++c)
        tmem_ld_32x32b_x32(taddr + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(v + 32 * c));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      // token j of the tile is row tc.m0 + j; 32 lanes write 64 contiguous bytes per row
      const int64_t rows = tc.m_end - tc.m0;
#pragma unroll
      for (int j = 0; j < C::TN; ++j) {
        if (j < rows) {
          float x = __uint_as_float(v[j]);
          if constexpr (C::POST != 1.0f) x *= C::POST;
          Cmat[(tc.m0 + j) * (int64_t)args.N + n] = __float2bfloat16_rn(x);
        }
      }
    }
  } else if (C::SF_ST && warp >= SFW_WARP0 && warp < SFW_WARP0 + 4) {
    // ============================== scale writers ===============================
    // Warp 8 + q stores TMEM lanes 32q..32q+31 of each stage's scale slot (the slot of stage
    // s is rewritten after the stage's loads of its next use landed, which followed the MMAs
    // that read the slot).  What the MMA reads there (pinned by the parity tests): for the
    // weights (its M operand) lane quarter q reads only column q of a 4-column group, row
    // 32q + i's codes at lane i; for the tokens (its N operand) every lane quarter reads
    // token row 32j + i's codes at lane i of column j, so each writer stores all token rows.
    const uint32_t q = warp & 3;
    GroupedScheduler<C::TN, WROWS> sched;
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    TileCoord tc;
    auto stage_ready = [&]() {
      if (!__all_sync(0xffffffffu, role_wait(full_bar(stage), phase, abort))) {
        if (lane == 0) record_error(args.err, DEV_TIMEOUT, abort);
        return false;
      }
      return true;
    };
    auto stage_done = [&]() {
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sfull_bar(stage));
      if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
    };
    if (sf_direct) {
      // Each lane fetches, STG_AHEAD groups of GS stages ahead, the 16-byte chunks of weight
      // row 32q + lane (unless the weight blocks come pre-packed with the stage) and of token
      // rows 32j + lane, into this warp's staging slots; nothing is shared between lanes.
      const uint8_t* a_sc = static_cast<const uint8_t*>(args.a_scales);
      const uint8_t* b_sc = static_cast<const uint8_t*>(args.b_scales);
      const int G = KB / GS;
      const uint32_t sWs = smem_u32(smem + C::SMEM_STG) + q * 512 + lane * 16;
      const uint32_t sTs = smem_u32(smem + C::SMEM_STGT) + q * (C::TN * 16) + lane * 16;
      const uint8_t* pWs = smem + C::SMEM_STG + q * 512 + lane * 16;
      const uint8_t* pTs = smem + C::SMEM_STGT + q * (C::TN * 16) + lane * 16;
      GroupedScheduler<C::TN, WROWS> pre;
      TileCoord tp;
      int64_t tp_t = blockIdx.x;
      bool pre_ok = pre.locate(args, tp_t, tp);
      int qp = 0;
      auto issue_group = [&](int slot) {
        if (pre_ok) {
          if (!packed_b)
            cp_async_16(sWs + slot * STG_SLOT,
                        b_sc + ((int64_t)tp.be * args.N + tp.n0 + 32 * q + lane) * scale_row +
                            16 * qp,
                        16u);
#pragma unroll
          for (int jt = 0; jt < C::TN / 32; ++jt) {
            const int64_t m = tp.m0 + 32 * jt + lane;
            const bool live = m < args.M_total;
            cp_async_16(sTs + slot * C::STGT_SLOT + jt * 512,
                        live ? a_sc + m * scale_row + 16 * qp : a_sc, live ? 16u : 0u);
          }
          if (++qp == G) {
            qp = 0;
            tp_t += gridDim.x;
            pre_ok = tp_t < total_tiles && pre.locate(args, tp_t, tp);
          }
        }
        cp_async_commit();  // an empty group keeps the group count in step
      };
      for (int a = 0; a < C::STG_AHEAD; ++a) issue_group(a);
      int64_t g = 0;
      for (int64_t t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
        if (!sched.locate(args, t, tc)) break;
        for (int qg = 0; ok && qg < G; ++qg, ++g) {
          cp_async_wait_group<C::STG_AHEAD - 1>();  // this lane's chunks of group g landed
          // the slot group g - 1 used is free (this lane read only its own chunks)
          issue_group((int)((g + C::STG_AHEAD) % C::STG_N));
          const uint32_t slot = (uint32_t)(g % C::STG_N);
          for (int j = 0; j < GS; ++j) {
            if (!stage_ready()) {
              ok = false;
              break;
            }
            const uint32_t tcol =
                tmem_base + ((q * 32) << 16) + C::ACC_COLS + stage * C::SF_STAGE_COLS;
#pragma unroll
            for (int b = 0; b < CPS / 4; ++b) {
              const uint32_t w =
                  packed_b ? *reinterpret_cast<const uint32_t*>(smem + C::SMEM_SFW +
                                                               stage * C::SFW_STAGE +
                                                               b * SF_BLOCK + lane * 16 + 4 * q)
                           : *reinterpret_cast<const uint32_t*>(pWs + slot * STG_SLOT +
                                                                CPS * j + 4 * b);
              tmem_st_32x32b_x1(tcol + 4 * b + q, w);
              // token rows 32 jt + lane at column jt of the group
              uint32_t x[C::TN / 32];
#pragma unroll
              for (int jt = 0; jt < C::TN / 32; ++jt)
                x[jt] = *reinterpret_cast<const uint32_t*>(pTs + slot * C::STGT_SLOT + jt * 512 +
                                                           CPS * j + 4 * b);
              if constexpr (C::TN >= 128)
                tmem_st_32x32b_x4(tcol + C::SF_COLS + 4 * b, x[0], x[1], x[2], x[3]);
              else if constexpr (C::TN >= 64)
                tmem_st_32x32b_x2(tcol + C::SF_COLS + 4 * b, x[0], x[1]);
              else
                tmem_st_32x32b_x1(tcol + C::SF_COLS + 4 * b, x[0]);
            }
            stage_done();
          }
        }
      }
      cp_async_wait_group<0>();
    } else {
      // relay: lane i takes the 16-byte row i of every packed 512-byte block (the loaders'
      // or the producer's) and writes it to 4 columns, as tcgen05.cp.32x128b.warpx4
      // replicates a block into all four lane quarters
      for (int64_t t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
        if (!sched.locate(args, t, tc)) break;
        for (int kb = 0; kb < KB; ++kb) {
          if (!stage_ready()) {
            ok = false;
            break;
          }
          const uint32_t tcol =
              tmem_base + ((q * 32) << 16) + C::ACC_COLS + stage * C::SF_STAGE_COLS;
#pragma unroll
          for (int b = 0; b < C::SF_GROUPS; ++b) {
            const uint4 w = *reinterpret_cast<const uint4*>(
                smem + C::SMEM_SFW + stage * C::SFW_STAGE + b * SF_BLOCK + lane * 16);
            const uint4 x = *reinterpret_cast<const uint4*>(
                smem + C::SMEM_SFT + stage * C::SFT_STAGE + b * SF_BLOCK + lane * 16);
            tmem_st_32x32b_x4(tcol + 4 * b, w.x, w.y, w.z, w.w);
            tmem_st_32x32b_x4(tcol + C::SF_COLS + 4 * b, x.x, x.y, x.z, x.w);
          }
          stage_done();
        }
      }
    }
  } else if (C::CONVERT && converter_index(warp) >= 0 && converter_index(warp) < C::NCONV) {
    // ================================ converters ================================
    // Slot c takes the stages i = c, c + CSTAGES, ... (counted over this CTA's tiles): load
    // slot i % STAGES into converted slot c, rows split among its SPLIT warps.  Before
    // reusing slot c a warp waits for the MMA's release of stage i - CSTAGES, the slot's
    // previous occupant (the commit on that stage's load-slot empty barrier), and only then
    // for stage i's loads: the MMA consumes in order, so by then the load slot's barrier is
    // in the phase of stage i.
    const int ci = converter_index(warp);
    const int c = ci / C::SPLIT, h = ci % C::SPLIT;
    GroupedScheduler<C::TN, WROWS> sched;
    int64_t i = 0;  // stage counter of this CTA
    bool ok = true;
    TileCoord tc;
    for (int64_t t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
      if (!sched.locate(args, t, tc)) break;
      for (int kb = 0; kb < KB; ++kb, ++i) {
        if (i % C::CSTAGES != c) continue;
        bool got = true;
        if (i >= C::CSTAGES) {
          const int64_t j = i - C::CSTAGES;
          got = role_wait(empty_bar((int)(j % C::STAGES)), (uint32_t)((j / C::STAGES) & 1),
                          abort);
        }
        const int stage = (int)(i % C::STAGES);
        if (got) got = role_wait(full_bar(stage), (uint32_t)((i / C::STAGES) & 1), abort);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) record_error(args.err, DEV_TIMEOUT, abort);
          ok = false;
          break;
        }
        if constexpr (C::NV_F16) {
          constexpr int WPART = WROWS / C::SPLIT, TPART = C::TN / C::SPLIT;
          convert_nvfp4_tile<WROWS, WPART>(smem + C::SMEM_W + stage * C::W_STAGE,
                                           smem + C::SMEM_SFW + stage * C::SFW_STAGE,
                                           smem + C::SMEM_CW + c * C::CW_STAGE, lane, h * WPART);
          convert_nvfp4_tile<C::TN, TPART>(smem + C::SMEM_T + stage * C::T_STAGE,
                                           smem + C::SMEM_SFT + stage * C::SFT_STAGE,
                                           smem + C::SMEM_CT + c * C::CT_STAGE, lane, h * TPART);
        } else {
          convert_fp4_tile<WROWS>(smem + C::SMEM_W + stage * C::W_STAGE,
                                  smem + C::SMEM_CW + c * C::CW_STAGE, lane);
          if constexpr (C::A_FP4)
            convert_fp4_tile<C::TN>(smem + C::SMEM_T + stage * C::T_STAGE,
                                    smem + C::SMEM_CT + c * C::CT_STAGE, lane);
        }
        fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads (async proxy)
        __syncwarp();
        if (lane == 0) mbar_arrive(cfull_bar(c));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<1>(tmem_base, C::TMEM_COLS);
  }
}

template <class C>
cudaError_t launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& args,
                   int num_sms, cudaStream_t stream) {
  static std::atomic<bool> attr_set[64];  // per device; several host threads may launch
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(bsmxfp8_kernel<C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes<C>());
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set[dev].store(true, std::memory_order_release);
  }
  const int64_t max_row_tiles = (args.M_total + C::TN - 1) / C::TN + args.E;
  const int64_t max_tiles = max_row_tiles * (args.N / WROWS);
  const int grid = (int)(max_tiles < num_sms ? max_tiles : num_sms);
  static_assert(smem_bytes<C>() <= SMEM_LIMIT, "shared memory");
  bsmxfp8_kernel<C><<<grid, C::THREADS, smem_bytes<C>(), stream>>>(tmA, tmB, args);
  return cudaGetLastError();
}

// One 512-byte block per iteration: thread r moves row r's 4 codes of the K block (one
// aligned 4-byte word of the row-major source) to byte (r % 32) * 16 + (r / 32) * 4.
__global__ void __launch_bounds__(128)
pack_b_scales_kernel(const uint8_t* src, uint8_t* dst, int64_t blocks, int KB, int scale_row) {
  const int r = (int)threadIdx.x;
  for (int64_t b = blockIdx.x; b < blocks; b += gridDim.x) {
    const int64_t kb = b % KB;
    const int64_t row = (b / KB) * WROWS + r;  // (e * N/128 + n block) * 128 + r = e * N + n
    const uint32_t w = *reinterpret_cast<const uint32_t*>(src + row * scale_row + 4 * kb);
    *reinterpret_cast<uint32_t*>(dst + b * SF_BLOCK + (r & 31) * 16 + (r >> 5) * 4) = w;
  }
}

}  // namespace mx

cudaError_t launch_pack_mx_b_scales(const uint8_t* src, uint8_t* dst, int E, int N, int K,
                                    int num_sms, cudaStream_t stream) {
  const int KB = K / mx::BK;
  const int64_t blocks = (int64_t)E * (N / mx::WROWS) * KB;
  if (blocks == 0) return cudaSuccess;
  const int64_t cap = (int64_t)num_sms * 16;
  const int grid = (int)(blocks < cap ? blocks : cap);
  mx::pack_b_scales_kernel<<<grid, 128, 0, stream>>>(src, dst, blocks, KB, K / 32);
  return cudaGetLastError();
}

cudaError_t launch_bsmxfp8(int tn, const CUtensorMap& tmA, const CUtensorMap& tmB,
                           const GemmArgs& args, int num_sms, cudaStream_t stream) {
  switch (tn) {
    case 32: return mx::launch<mx::Cfg<32>>(tmA, tmB, args, num_sms, stream);
    case 64: return mx::launch<mx::Cfg<64>>(tmA, tmB, args, num_sms, stream);
    case 128: return mx::launch<mx::Cfg<128>>(tmA, tmB, args, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

// fp4 operands: a_fp4 = tokens packed e2m1 (else e4m3); the weights are packed e2m1; tn is
// 32 or 64 (and 128 with mma_kind).  mma_kind: kind::mxf4 on the packed tiles, stage_k K per stage (a_fp4), or
// kind::mxf8f6f4 on e2m1 weight tiles loaded padded (e4m3 tokens).
cudaError_t launch_bsmxfp4(int tn, bool a_fp4, bool mma_kind, int stage_k, const CUtensorMap& tmA,
                           const CUtensorMap& tmB, const GemmArgs& args, int num_sms,
                           cudaStream_t stream) {
  using namespace mx;
  if (!a_fp4 && mma_kind && stage_k == 256) {
    switch (tn) {
      case 32: return launch<Cfg<32, FMT_MXFP8_MXFP4_MMA, 256>>(tmA, tmB, args, num_sms, stream);
      case 64: return launch<Cfg<64, FMT_MXFP8_MXFP4_MMA, 256>>(tmA, tmB, args, num_sms, stream);
    }
  } else if (!a_fp4 && mma_kind) {
    switch (tn) {
      case 32: return launch<Cfg<32, FMT_MXFP8_MXFP4_MMA>>(tmA, tmB, args, num_sms, stream);
      case 64: return launch<Cfg<64, FMT_MXFP8_MXFP4_MMA>>(tmA, tmB, args, num_sms, stream);
      case 128: return launch<Cfg<128, FMT_MXFP8_MXFP4_MMA>>(tmA, tmB, args, num_sms, stream);
    }
  } else if (a_fp4 && mma_kind && stage_k == 256) {
    switch (tn) {
      case 32: return launch<Cfg<32, FMT_MXFP4_MMA, 256>>(tmA, tmB, args, num_sms, stream);
      case 64: return launch<Cfg<64, FMT_MXFP4_MMA, 256>>(tmA, tmB, args, num_sms, stream);
      case 128: return launch<Cfg<128, FMT_MXFP4_MMA, 256>>(tmA, tmB, args, num_sms, stream);
    }
  } else if (a_fp4 && mma_kind) {
    switch (tn) {
      case 32: return launch<Cfg<32, FMT_MXFP4_MMA>>(tmA, tmB, args, num_sms, stream);
      case 64: return launch<Cfg<64, FMT_MXFP4_MMA>>(tmA, tmB, args, num_sms, stream);
      case 128: return launch<Cfg<128, FMT_MXFP4_MMA>>(tmA, tmB, args, num_sms, stream);
    }
  } else if (a_fp4) {
    switch (tn) {
      case 32: return launch<Cfg<32, FMT_MXFP4>>(tmA, tmB, args, num_sms, stream);
      case 64: return launch<Cfg<64, FMT_MXFP4>>(tmA, tmB, args, num_sms, stream);
    }
  } else {
    switch (tn) {
      case 32: return launch<Cfg<32, FMT_MXFP8_MXFP4>>(tmA, tmB, args, num_sms, stream);
      case 64: return launch<Cfg<64, FMT_MXFP8_MXFP4>>(tmA, tmB, args, num_sms, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace bsfp8

namespace bsfp8 {
// nvfp4 x nvfp4: both operands packed e2m1 with e4m3 scales per 16 K; tn is 32 or 64.
// mma_kind: kind::mxf4nvf4 (scale_vec::4X) on the packed tiles.
cudaError_t launch_bsnvfp4(int tn, bool mma_kind, int stage_k, const CUtensorMap& tmA,
                           const CUtensorMap& tmB, const GemmArgs& args, int num_sms,
                           cudaStream_t stream) {
  using namespace mx;
  if (mma_kind && stage_k == 256) {
    switch (tn) {
      case 32: return launch<Cfg<32, FMT_NVFP4_MMA, 256>>(tmA, tmB, args, num_sms, stream);
      case 64: return launch<Cfg<64, FMT_NVFP4_MMA, 256>>(tmA, tmB, args, num_sms, stream);
      case 128: return launch<Cfg<128, FMT_NVFP4_MMA, 256>>(tmA, tmB, args, num_sms, stream);
    }
    return cudaErrorInvalidValue;
  }
  if (mma_kind) {
    switch (tn) {
      case 32: return launch<Cfg<32, FMT_NVFP4_MMA>>(tmA, tmB, args, num_sms, stream);
      case 64: return launch<Cfg<64, FMT_NVFP4_MMA>>(tmA, tmB, args, num_sms, stream);
      case 128: return launch<Cfg<128, FMT_NVFP4_MMA>>(tmA, tmB, args, num_sms, stream);
    }
    return cudaErrorInvalidValue;
  }
  switch (tn) {
    case 32: return launch<Cfg<32, FMT_NVFP4>>(tmA, tmB, args, num_sms, stream);
    case 64: return launch<Cfg<64, FMT_NVFP4>>(tmA, tmB, args, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}
}  // namespace bsfp8

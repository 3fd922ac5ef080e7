/*
 * bsfp8 -- blockwise-scaled FP8 grouped GEMM for GB300 (sm_103a), C ABI.
 *
 * The operation (mixture-of-experts grouped GEMM with blockwise FP8 scaling):
 *
 *   for every expert e, every row m in [expert_offsets[e], expert_offsets[e+1]) and every
 *   column n < N:
 *     C[m, n] = bf16( sum_kb  sa(m, kb) * sb(e, n, kb) * sum_{k in block kb} A[m, k] * B[e, n, k] )
 *
 *   A, B are e4m3 ("fn") codes; the inner sums run over K blocks; accumulation is fp32 and
 *   the result is rounded to bf16 (round to nearest even).
 *
 * Sources (the pages this library follows):
 *   - promote_accumulators (MAX kernels, linalg/grouped_matmul_sm100_blockwise_fp8),
 *     description and Args: each per-K-block MMA result is multiplied by the A scale of
 *     its row and the B scale of its (expert, N block, K block) and accumulated in fp32
 *     register tiles; b_scales has shape [num_experts, N // BN, K // BK]; problem_shape
 *     is (M, N, K); expert_ids maps a group to its expert's rows of B.
 *   - EpilogueWarpContext (MAX sm100_structured warp_context), per_k_stage: the blockwise
 *     FP8 epilogue consumes one TMEM stage and one A-scale stage per K iteration.
 *   - Triton Gluon example "Overlapping Accumulator Block-Scaled Matrix Multiplication",
 *     async_mma_scaled_impl / random_quantized_tensor / swizzle_scales_packed_block: the
 *     block-scaled MMA on e4m3 operands with UE8M0 (uint8) scales, one per VEC_SIZE = 32
 *     elements of K, the scales arranged in 128-row packed blocks for the tensor core.
 *
 * Conventions shared by every entry point:
 *   - Every pointer is a DEVICE pointer (memory of the current CUDA device), row-major,
 *     last index contiguous.  The caller owns every buffer and the stream; the library
 *     keeps only a 4-byte device error word per device and allocates nothing per call.
 *   - Calls are asynchronous and ordered on `stream`; nothing is synchronised.
 *   - Host-detectable problems return a status immediately and launch nothing.
 *   - Problems only the device can see (expert offsets that are not a valid partition of
 *     [0, M_total), or a pipeline wait that exceeded its time limit) make the kernel write
 *     a code into the device error word and finish without touching C further; read it
 *     with bsfp8_get_device_error().
 *   - Requirements: N % 128 == 0, K % 128 == 0, num_experts >= 1, 0 <= M_total < 2^31,
 *     num_experts * N < 2^31; A, B, C 16-byte aligned; scales and offsets 4-byte aligned
 *     (also the UE8M0 scale arrays, which are read 4 codes at a time).  A 32-byte aligned C
 *     is written with 32-byte stores (faster), a 16-byte aligned one with 16-byte stores.
 *     M_total == 0 is a valid no-op (nothing is read or written).
 *   - The device must be compute capability 10.3 (GB300).
 */
#ifndef BSFP8_H_
#define BSFP8_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#ifndef __CUDA_RUNTIME_API_H__
/* Same type as the CUDA runtime's cudaStream_t. */
typedef struct CUstream_st* cudaStream_t;
#endif

typedef enum {
  BSFP8_OK = 0,
  BSFP8_ERR_NULL = 1,               /* a required pointer is NULL */
  BSFP8_ERR_SHAPE = 2,              /* sizes violate the requirements above */
  BSFP8_ERR_ALIGN = 3,              /* a pointer is not aligned as required */
  BSFP8_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not compute capability 10.3 */
  BSFP8_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed (launch, ...) */
  BSFP8_ERR_DEVICE_OFFSETS = 6,     /* device error word: invalid expert offsets */
  BSFP8_ERR_DEVICE_TIMEOUT = 7,     /* device error word: a pipeline wait gave up */
  BSFP8_ERR_DEVICE_EXPERT_IDS = 8,  /* device error word: an expert id outside [0, num_experts) */
  BSFP8_ERR_FORMAT = 9,             /* bsmx_grouped_gemm: unsupported operand format pair */
  BSFP8_ERR_DEVICE_BOUNDS = 10      /* device error word, debug builds only: a tile's rows,
                                       columns or expert fell outside the problem */
} bsfp8_status;

/* Operand formats of bsmx_grouped_gemm. */
typedef enum {
  BSMX_MXFP8 = 0, /* e4m3 elements, one byte each;        UE8M0 scale per 32 elements of K */
  BSMX_MXFP4 = 1, /* e2m1 elements, two per byte along K; UE8M0 scale per 32 elements of K */
  BSMX_NVFP4 = 2  /* e2m1 elements, two per byte along K; e4m3 scale per 16 elements of K */
} bsmx_format;

/*
 * Blockwise FP8 grouped GEMM (1x128 A scales, 128x128 B scales).
 *
 *   A              e4m3 [M_total, K]        token rows, grouped by expert (expert e owns
 *                                           rows expert_offsets[e] .. expert_offsets[e+1]-1)
 *   B              e4m3 [num_experts, N, K] expert weights, K-major (row n of expert e is
 *                                           B + (e*N + n)*K)
 *   a_scales       fp32 [K/128, M_total]    sa(m, kb) = a_scales[kb*M_total + m]
 *   b_scales       fp32 [num_experts, N/128, K/128]
 *                                           sb(e, n, kb) = b_scales[(e*(N/128) + n/128)*(K/128) + kb]
 *   expert_offsets int32 [num_experts+1]    expert_offsets[0] = 0, non-decreasing,
 *                                           expert_offsets[num_experts] = M_total
 *   C              bf16 [M_total, N]        output, fully written (every row belongs to
 *                                           exactly one expert); experts with no rows
 *                                           write nothing
 */
bsfp8_status bsfp8_grouped_gemm(const void* A, const void* B, const float* a_scales,
                                const float* b_scales, const int32_t* expert_offsets, void* C,
                                int64_t M_total, int N, int K, int num_experts,
                                cudaStream_t stream);

/*
 * MXFP8 grouped GEMM: e4m3 operands, UE8M0 scales (2^(code-127)) per 32 elements of K,
 * applied by the block-scaled tensor-core MMA:
 *
 *   C[m, n] = bf16( sum_k A[m,k] * B[e,n,k] * 2^(a_scales[m, k/32] - 127) * 2^(b_scales[e, n, k/32] - 127) )
 *
 *   A              e4m3 [M_total, K]             token rows, grouped by expert
 *   B              e4m3 [num_experts, N, K]      expert weights, K-major
 *   a_scales       UE8M0 [M_total, K/32]         row-major (row m's codes are contiguous)
 *   b_scales       UE8M0 [num_experts, N, K/32]  row-major
 *   expert_offsets int32 [num_experts+1]         as for bsfp8_grouped_gemm
 *   C              bf16 [M_total, N]             output
 *
 * Same requirements, ownership and error behaviour as bsfp8_grouped_gemm.  Tile forms:
 * "swap-AB" tiles pair 128 rows of an expert's weights with up to 32 / 64 / 128 of its token
 * rows (the height follows M_total / num_experts); CTA-pair 256 x 256 tiles have overlapping
 * double-buffered TMEM accumulators.  With at most 24 token rows per expert on average the
 * call runs swap-AB tiles, above 56 the CTA-pair tiles, and in between both kernels one after
 * the other on `stream`: experts with at least 256 rows on the CTA-pair tiles, the others on
 * swap-AB tiles of 64 token rows, each kernel writing its own experts' rows of C (the
 * per-expert counts are only known on the device).  Environment variables override the
 * choice: BSFP8_MX_KERNEL = swap | pair | split, BSFP8_MX_TN = 32 | 64 | 128 (swap-AB
 * height).  Every form meets the same accuracy bound.
 */
bsfp8_status bsmxfp8_grouped_gemm(const void* A, const void* B, const uint8_t* a_scales,
                                  const uint8_t* b_scales, const int32_t* expert_offsets,
                                  void* C, int64_t M_total, int N, int K, int num_experts,
                                  cudaStream_t stream);

/*
 * The same two GEMMs with an expert indirection: the rows of A form num_groups groups
 * (group g owns rows group_offsets[g] .. group_offsets[g+1]-1) and group g multiplies the
 * weights of expert expert_ids[g] -- its rows of B and of b_scales -- instead of expert g.
 * This is the expert_ids argument of promote_accumulators (MAX kernels,
 * grouped_matmul_sm100_blockwise_fp8, Args: "mapping from group index to expert row offset
 * in B"): only the experts that received tokens need a group, and several groups may use the
 * same expert.
 *
 *   group_offsets  int32 [num_groups+1]  as expert_offsets above, per group
 *   expert_ids     int32 [num_groups]    device array, each in [0, num_experts)
 *   B, b_scales    as above, with num_experts experts
 *   A, a_scales, C as above (M_total rows)
 *
 *   C[m, n] = bf16( sum_kb sa(m, kb) * sb(x, n, kb) * sum_{k in kb} A[m,k] * B[x,n,k] ),
 *             x = expert_ids[g] for the group g that owns row m (blockwise; the MXFP8 entry
 *             point applies its UE8M0 scales the same way)
 *
 * expert_ids may not be NULL (BSFP8_ERR_NULL); num_groups >= 1 and num_experts >= 1
 * (BSFP8_ERR_SHAPE); expert_ids 4-byte aligned.  An id outside [0, num_experts) is found on the
 * device: the kernel writes nothing, records BSFP8_ERR_DEVICE_EXPERT_IDS in the device error
 * word and finishes.  Everything else (requirements, ownership, asynchrony) is as for the
 * entry points without ids, which are these with expert_ids[g] = g and num_groups =
 * num_experts.
 */
bsfp8_status bsfp8_grouped_gemm_ids(const void* A, const void* B, const float* a_scales,
                                    const float* b_scales, const int32_t* group_offsets,
                                    const int32_t* expert_ids, void* C, int64_t M_total, int N,
                                    int K, int num_groups, int num_experts, cudaStream_t stream);

bsfp8_status bsmxfp8_grouped_gemm_ids(const void* A, const void* B, const uint8_t* a_scales,
                                      const uint8_t* b_scales, const int32_t* group_offsets,
                                      const int32_t* expert_ids, void* C, int64_t M_total, int N,
                                      int K, int num_groups, int num_experts,
                                      cudaStream_t stream);

/*
 * Pre-packed MXFP8 weight scales.  Expert weights are static, so their UE8M0 scales can be
 * rearranged once into the tensor core's scale-factor layout, which the GEMM then copies
 * straight into shared memory instead of gathering and transposing 4 codes per row per
 * K block.  The layout is the 128-row "packed block" of swizzle_scales_packed_block in the
 * Triton Gluon example "Overlapping Accumulator Block-Scaled Matrix Multiplication" (rows
 * padded to 128 and scale columns to 4, viewed as (rows/128, 4, 32, cols/4, 4) and permuted
 * (0, 3, 2, 1, 4)); here N % 128 == 0 and K % 128 == 0, so nothing is padded:
 *
 *   b_scales_packed  UE8M0 [num_experts, N/128, K/128, 512]
 *     byte (r % 32) * 16 + (r / 32) * 4 + j of block (e, nb, kb) =
 *     b_scales[e, nb*128 + r, 4*kb + j]          (r < 128, j < 4)
 *
 * bsmxfp8_pack_b_scales writes it (num_experts * N * K/32 bytes, the size of the source)
 * on `stream`; b_scales 4-byte aligned, b_scales_packed 16-byte aligned.  Errors:
 * BSFP8_ERR_NULL, BSFP8_ERR_SHAPE (num_experts >= 1, N and K multiples of 128,
 * num_experts * N < 2^31), BSFP8_ERR_ALIGN, BSFP8_ERR_UNSUPPORTED_DEVICE, BSFP8_ERR_CUDA.
 *
 * bsmxfp8_grouped_gemm_prepacked is bsmxfp8_grouped_gemm with b_scales_packed (16-byte
 * aligned) in place of b_scales, on the kernel the plan picks: swap-AB tiles (128 weight rows
 * = one packed block per K block) or CTA-pair 256 x 256 tiles (two blocks per K block).  Same
 * result, requirements and errors otherwise.
 */
bsfp8_status bsmxfp8_pack_b_scales(const uint8_t* b_scales, uint8_t* b_scales_packed,
                                   int num_experts, int N, int K, cudaStream_t stream);

bsfp8_status bsmxfp8_grouped_gemm_prepacked(const void* A, const void* B, const uint8_t* a_scales,
                                            const uint8_t* b_scales_packed,
                                            const int32_t* expert_offsets, void* C,
                                            int64_t M_total, int N, int K, int num_experts,
                                            cudaStream_t stream);

/*
 * Block-scaled grouped GEMM with a format per operand: the formats and format pairs of the
 * Triton Gluon example "Overlapping Accumulator Block-Scaled Matrix Multiplication"
 * (Fixed Configuration, FORMATS; random_quantized_tensor: scales per VEC_SIZE = 32 K
 * elements as uint8 UE8M0, or per 16 as float8_e4m3fn for nvfp4; fp4 elements packed along
 * K, stored as uint8 and read by the MMA as "e2m1").
 *
 *   A          [M_total, K] elements in a_format: K bytes per row (MXFP8) or K/2 (fp4: element
 *              2i of the row in the low nibble of byte i, element 2i+1 in the high nibble)
 *   B          [num_experts, N, K] elements in b_format, laid out the same way
 *   a_scales   [M_total, K/vec] codes (vec = 32: UE8M0; vec = 16 for NVFP4: unsigned e4m3,
 *              codes 0x00..0x7E, bit 7 zero: the example draws them positive), row-major
 *   b_scales   [num_experts, N, K/vec] codes, row-major; with b_scales_packed != 0 (MXFP8 and
 *              MXFP4 weights only) the 512-byte block layout of bsmxfp8_pack_b_scales,
 *              16-byte aligned
 *   group_offsets, C, M_total, N, K, num_groups, num_experts, stream
 *              as for bsmxfp8_grouped_gemm_ids; expert_ids as there, or NULL for group g ->
 *              expert g (then num_groups must equal num_experts: BSFP8_ERR_SHAPE)
 *
 *   C[m, n] = bf16( sum_k dec(A[m,k]) * sa(m, k/vec_a) * dec(B[x,n,k]) * sb(x, n, k/vec_b) ),
 *             x the expert of row m's group
 *
 * Supported (a_format, b_format) pairs:
 *   (MXFP8, MXFP8)  bsmxfp8_grouped_gemm(_ids) / _prepacked
 *   (MXFP4, MXFP4)  swap-AB tiles at every size; the packed tiles feed the fp4 block-scaled
 *                   MMA (tcgen05.mma kind::mxf4, K = 64 per instruction, UE8M0 per 32) as
 *                   loaded.  Every product is taken exactly and summed in fp32.
 *   (NVFP4, NVFP4)  swap-AB tiles at every size; the packed tiles feed tcgen05.mma
 *                   kind::mxf4nvf4 with scale_vec::4X (UE4M3 per 16) as loaded.  The scales
 *                   must be 8-byte aligned (BSFP8_ERR_ALIGN); b_scales_packed is not
 *                   available (BSFP8_ERR_FORMAT).  A scale code with bit 7 set is outside the
 *                   format (the tensor core's scale type is unsigned): its result is not
 *                   specified.
 *   (MXFP8, MXFP4)  swap-AB tiles at every size; tcgen05.mma kind::mxf8f6f4 with e4m3 tokens
 *                   and e2m1 weights (K = 32 per instruction, UE8M0 per 32), the packed
 *                   weight tiles landing in shared memory padded (a byte per element) as
 *                   the tensor memory access unit expands them.  B must be 32-byte aligned
 *                   for that load; a B that is only 16-byte aligned runs the converting form.
 * Stages of 256 K run where every scale row's codes come in aligned 16-byte chunks (K % 512
 * == 0 for the mx formats, K % 256 for nvfp4, a_scales and b_scales 16-byte aligned), else
 * stages of 128 K; environment variable BSFP8_FP4_STAGE_K=128 keeps 128 K.  Prefill-sized
 * batches (more than 128 token rows per row group on average; BSFP8_MX_KERNEL = pair | swap
 * overrides) run the
 * CTA-pair 256 x 256 kernel on the same MMA kinds: mxfp8 x mxfp4 with a 32-byte aligned B,
 * the fp4 x fp4 pairs on chunkable scale rows with row-major weight scales; other batches
 * run the swap-AB tiles.  Results do not depend on these choices.
 * Converting forms (environment variable BSFP8_FP4_MMA=convert selects them for every pair;
 * kept for comparison):
 *   MX pairs        the packed tiles are re-encoded on chip into e4m3 for the MXFP8
 *                   block-scaled MMA: every e2m1 value times 2^-6 is an e4m3 value, and the
 *                   epilogue multiplies the fp32 sums by 2^6 per fp4 operand, so the result
 *                   is that of the same values in MXFP8 while the tensor core's products,
 *                   2^-6 per fp4 operand below the true ones, stay in fp32's normal range:
 *                   every non-zero product dec(A)*sa*dec(B)*sb of magnitude at least 2^-120
 *                   (one fp4 operand) or 2^-114 (two).  Smaller products may be flushed to
 *                   zero.
 *   NVFP4           the packed tiles and their e4m3 scales are dequantized on chip into
 *                   fp16 (exact: an e2m1 value times an e4m3 scale has at most 6 significant
 *                   bits and lies in the normal fp16 range) and multiplied by the fp16
 *                   tensor-core MMA with fp32 accumulation.
 * Any other pair returns BSFP8_ERR_FORMAT with nothing launched.  Requirements, ownership,
 * asynchrony and the other errors are those of bsmxfp8_grouped_gemm_ids (A, B and C 16-byte
 * aligned; N and K multiples of 128).
 */
bsfp8_status bsmx_grouped_gemm(int a_format, int b_format, const void* A, const void* B,
                               const uint8_t* a_scales, const uint8_t* b_scales,
                               int b_scales_packed, const int32_t* group_offsets,
                               const int32_t* expert_ids, void* C, int64_t M_total, int N, int K,
                               int num_groups, int num_experts, cudaStream_t stream);

/*
 * TMEM storage plan of double-buffered block-scaled accumulators (host only, no GPU use).
 * For a 256-column tile with 512 TMEM columns, block_k elements of K per MMA stage,
 * epilogue subtiles of epilogue_n columns and one scale per vec (16 or 32) elements of K,
 * writes into out[9]: left accumulator offset and columns, right accumulator offset and
 * columns, A-scale offset and columns, B-scale offset and columns, and the epilogue
 * subtile that holds the overlapped columns.  With overlap != 0 the second accumulator
 * overlaps the first by the scale columns (the Overlapping Accumulator Layout section and
 * tmem_overlap_storage_plan of the Triton Gluon example "Overlapping Accumulator
 * Block-Scaled Matrix Multiplication"); with overlap == 0 a single accumulator is
 * followed by the scales.  block_k == 0 returns the plan the CTA-pair MXFP8 kernel of
 * bsmxfp8_grouped_gemm is compiled with.  BSFP8_ERR_NULL / BSFP8_ERR_SHAPE on bad input.
 */
bsfp8_status bsmxfp8_tmem_plan(int block_k, int epilogue_n, int vec, int overlap, int32_t* out);

/*
 * Tile plan bsfp8_grouped_gemm uses for a problem of this size on a device with num_sms SMs
 * (host only, no GPU use; BSFP8_BLOCKWISE_TILE is honoured as in the GEMM): writes out[0] =
 * tile rows, out[1] = tile columns, out[2] = CTAs per tile (1, or 2 for a CTA pair).  The
 * persistent kernel gives each CTA (pair) every (SMs / CTAs per tile)-th tile; tiles are
 * ceil(M_e / rows) x ceil(N / columns) per expert e.  The default picks 96 x 256 tiles on
 * one CTA, 192 x 256 on a CTA pair or 224 x 256 on an asymmetric pair (a 96-row CTA with the
 * producer and MMA warps next to a 128-row CTA of epilogue warps only) by estimated makespan.
 * This is a performance choice only: every plan computes the same result.  The environment
 * variable BSFP8_BLOCKWISE_TILE names a tile form for the GEMM to use instead (cta1_96,
 * pair_192, pair_224, cta1_256, pair_256, ...), or "split": groups with at least
 * BSFP8_BLOCKWISE_SPLIT_ROWS rows (default 448) on 224 x 256 pair tiles, then the others on
 * 96 x 256 tiles, as two kernels on the GEMM's stream; this function then reports the default
 * plan.  BSFP8_ERR_NULL / BSFP8_ERR_SHAPE on bad input.
 */
bsfp8_status bsfp8_blockwise_plan(int64_t M_total, int N, int num_experts, int num_sms,
                                  int32_t* out);

/*
 * Kernel plan bsmxfp8_grouped_gemm (and its _ids / _prepacked forms) uses for M_total token
 * rows over num_experts row groups (host only, no GPU use; BSFP8_MX_KERNEL and BSFP8_MX_TN
 * are honoured as in the GEMM): out[0] = 0 for swap-AB tiles, 1 for CTA-pair 256 x 256 tiles,
 * 2 for both (split by rows per group); out[1] = token rows per swap-AB tile (0 when only the
 * CTA-pair kernel runs); out[2] = the split's row threshold (groups with at least this many
 * rows run on the CTA-pair tiles; 0 without a split).  A performance choice only: every plan
 * meets the same accuracy bound.  BSFP8_ERR_NULL / BSFP8_ERR_SHAPE on bad input.
 */
bsfp8_status bsmxfp8_plan(int64_t M_total, int num_experts, int32_t* out);

/*
 * Tile form bsmx_grouped_gemm (and its _ids form) uses for M_total token rows over
 * num_groups row groups (host only, no GPU use; BSFP8_MX_KERNEL, BSFP8_MX_TN and
 * BSFP8_FP4_MMA are honoured as in the GEMM): out[0] = 1 for CTA-pair 256 x 256 tiles (more
 * than 128 rows per group on average, on the fp4 MMA kinds), 0 for swap-AB tiles; out[1] =
 * token rows per swap-AB tile (32, 64 or 128; at most 64 on the converting forms; 0 with
 * CTA-pair tiles).  The GEMM takes the CTA-pair tiles only where the operands also meet their
 * conditions (mxfp8 x mxfp4: B 32-byte aligned; fp4 x fp4: row-major weight scales, K % 512
 * == 0 for mxfp4 or K % 256 for nvfp4, 16-byte aligned scales), else swap-AB tiles.  A
 * performance choice only.  BSFP8_ERR_NULL / BSFP8_ERR_SHAPE on bad input.
 */
bsfp8_status bsmx_plan(int64_t M_total, int num_groups, int32_t* out);

/*
 * Read the device error word of the current device (after synchronising `stream`) into
 * *code (0, BSFP8_ERR_DEVICE_OFFSETS, BSFP8_ERR_DEVICE_TIMEOUT, BSFP8_ERR_DEVICE_EXPERT_IDS, or
 * in a debug build BSFP8_ERR_DEVICE_BOUNDS)
 * and reset it to 0.
 * The word is one per device, not per stream: every kernel of this library on the device
 * records its first error there, whatever stream it runs on.  Only `stream` is synchronised,
 * so a kernel still running on another stream can set the word after it is read, or have its
 * error read (and cleared) by this call on behalf of the wrong caller.  Callers that launch on
 * several streams synchronise the device (cudaDeviceSynchronize) before reading the word.
 * Returns BSFP8_ERR_NULL for a NULL code, BSFP8_ERR_CUDA if a CUDA call fails.
 */
bsfp8_status bsfp8_get_device_error(cudaStream_t stream, int* code);

/*
 * Failure-detection check (no GEMM): launches one thread on `stream` that waits, with the
 * same bounded mbarrier wait every pipeline stage of the GEMM kernels uses, for a barrier
 * phase that nothing completes.  After limit_ns nanoseconds of %globaltimer (0 < limit_ns
 * <= 1e9; the GEMM kernels use 1 s) the wait gives up, BSFP8_ERR_DEVICE_TIMEOUT is recorded
 * in the device error word -- read it with bsfp8_get_device_error() -- and the kernel
 * returns, leaving the context usable.  Nothing else is read or written.
 * BSFP8_ERR_SHAPE for a limit out of range, BSFP8_ERR_UNSUPPORTED_DEVICE, BSFP8_ERR_CUDA.
 */
bsfp8_status bsfp8_check_wait_timeout(int64_t limit_ns, cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char* bsfp8_status_string(bsfp8_status status);

#ifdef __cplusplus
}
#endif

#endif /* BSFP8_H_ */

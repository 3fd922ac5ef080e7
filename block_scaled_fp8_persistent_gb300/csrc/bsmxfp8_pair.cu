// MXFP8 grouped GEMM with CTA-pair 256 x 256 tiles and overlapping double-buffered TMEM
// accumulators (for experts with many token rows).
//
//   C[m, n] = sum_k A[m,k] * B[e,n,k] * 2^(a_scales[m, k/32] - 127) * 2^(b_scales[e, n, k/32] - 127)
//
// Prior art: the Triton Gluon example "Overlapping Accumulator Block-Scaled Matrix
// Multiplication" (2-CTA block-scaled MMA, BLOCK_M = BLOCK_N = 256, the Overlapping
// Accumulator Layout section, tmem_overlap_storage_plan, the mma / epilogue partitions and
// the overlap barrier).  Differences: tiles walk expert segments; each CTA loads its own
// operand halves (no multicast); scales arrive row-major and are packed on chip by a
// loader warp; bf16 output.
//
// TMEM (512 columns per CTA, plan for BLOCK_K = 128, VEC = 32):
//   left accumulator  [0, 256)     even tiles
//   right accumulator [244, 500)   odd tiles (overlaps the left one in 12 columns)
//   A scales          [500, 504)   this CTA's 128 token rows
//   B scales          [504, 512)   all 256 weight rows of the tile (both 128-row blocks)
// An even tile's epilogue drains high columns first, an odd tile's low columns first, so
// the overlapped columns are read first; the warps holding them then arrive on the
// overlap barrier and the next tile's MMA (into the other accumulator) may start, while
// the MMA two tiles later waits for the whole accumulator (acc_empty).
//
// Roles (12 warps per CTA; 16 for the fp4 x fp4 forms): warp 0 TMA producer (own 128 token
// rows, own 128 weight rows); warp 1 TMEM owner and, in CTA 0 of the pair, the MMA thread
// (per 128-K block tcgen05.cp of its scale blocks and 4 x
// tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale; one commit per ring stage, multicast
// to both CTAs); warp 2 scale loader (fp4 x fp4: warps 2 and 3, alternate chunk groups);
// warps 4-11 epilogue (TMEM lane quarter w%4, column half (w-4)/4, 32-column subtiles);
// fp4 x fp4: warps 12-15 scale writers (tcgen05.st into the plan's scale slots, so the MMA
// thread issues only MMAs and commits).
// A ring stage holds KG = 2 K blocks (the k_group_size grouping of K iterations per
// pipeline stage): the full/empty barriers, the scale announce and the commit are paid once
// per 256 of K.
#include <atomic>
#include <cuda_bf16.h>
#include "common.cuh"
#include "ptx.cuh"
#include "sched.cuh"
#include "tmem_plan.cuh"

namespace bsfp8 {
namespace mxp {

// tcgen05.st of 8 consecutive 32-bit columns per lane (the writer warps' weight-scale words)
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                   taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

constexpr int BK = 128;
constexpr int BM = 256;        // token rows per pair tile (128 per CTA)
constexpr int BN = 256;        // weight rows per pair tile (MMA N)
constexpr int EPI_N = 32;      // epilogue subtile columns
// Tiles are walked in bands of 16 row tiles (row index fastest inside a band): the 76 pairs
// in flight share ~5 columns of B, and B is read from DRAM about once per band
constexpr int TILE_BAND = 16;
constexpr int NUM_THREADS = 384;  // the MXFP8 forms' block (PCfg::THREADS per form)
constexpr int EPI_WARP0 = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr int SF_BLOCK = 512;  // packed scale block: 128 rows x 4 codes
// Operand formats (A = tokens, B = weights): MXFP8 e4m3 x e4m3; MIXED e4m3 x e2m1 (the weights
// loaded padded, a byte per element, for kind::mxf8f6f4); MXF4 e2m1 x e2m1 (kind::mxf4, UE8M0
// per 32); NVF4 e2m1 x e2m1 with UE4M3 scales per 16 (kind::mxf4nvf4, scale_vec::4X).
enum PairFormat : int { PF_MXFP8 = 0, PF_MIXED = 1, PF_MXF4 = 2, PF_NVF4 = 3 };

template <int FMT_>
struct PCfg {
  static constexpr int FMT = FMT_;
  static constexpr bool FP4 = FMT_ >= PF_MXF4;  // both operands packed e2m1
  // K per K block: a 128-byte row of the operand tile (128 e4m3 or padded e2m1, 256 packed
  // e2m1), four MMAs (K = 32, or K = 64 for the fp4 kinds)
  static constexpr int KBLK = FP4 ? 256 : 128;
  static constexpr int VEC = FMT_ == PF_NVF4 ? 16 : 32;  // K per scale code
  static constexpr int CPK = KBLK / VEC;  // scale codes per row and K block: 4, 8 or 16
  static constexpr int G = CPK / 4;       // 4-column TMEM scale groups per 128 rows
  // K blocks per ring stage (the k_group_size grouping of K iterations per pipeline stage,
  // MAX EpilogueWarpContext page, per_k_stage): one full/empty round trip and one commit
  // per KG K blocks
  static constexpr int KG = FP4 ? 1 : 2;
  static constexpr int STAGES = FP4 ? 5 : 3;  // ring stages (64 or 32 KB of operands each)
  // scale loader warps per CTA: the fp4 x fp4 forms, with 2 or 4 scale groups per K block,
  // take alternate chunk groups (below; warp 2 the even ones, warp 3 the odd ones), each
  // fetching and transposing all rows of its own groups, so that one loader per CTA
  // announces each stage
  static constexpr int LOADERS = FP4 ? 2 : 1;
  // Scale feed.  MXFP8 forms: the MMA thread copies each K block's blocks into the plan's
  // scale columns (tcgen05.cp), in issue order after the previous K block's MMAs.  fp4 x fp4
  // forms (SF_ST): SF_SLOTS scale slots, K block i in slot i % SF_SLOTS, stored
  // (tcgen05.st) by four writer warps per CTA (one per TMEM lane quarter) from the loaders'
  // packed blocks ahead of the MMAs.  The plan is that of a K block SF_SLOTS times as long:
  // the two accumulators overlap by all the slots, which must stay inside the column half
  // whose epilogue warps release the overlap (mxfp4: three slots, 72 columns; nvfp4: two,
  // 96 columns, as three would take 144).
  static constexpr bool SF_ST = FP4;
  static constexpr int THREADS = SF_ST ? 512 : 384;
  static constexpr int SF_SLOTS = FMT_ == PF_MXF4 ? 3 : (FMT_ == PF_NVF4 ? 2 : 1);
  static constexpr TmemPlan PLAN =
      tmem_overlap_plan(SF_SLOTS * KBLK, EPI_N, VEC, true, BN, 512);
  static constexpr int SFA_COLS = 4 * G;  // one slot's token-scale columns
  static constexpr int SFB_COLS = 8 * G;  // one slot's weight-scale columns
  static constexpr uint32_t A_SUB = 128 * 128;  // one K block of this CTA's token rows
  static constexpr uint32_t B_SUB = 128 * 128;  // one K block of this CTA's weight rows
  static constexpr uint32_t A_STAGE = KG * A_SUB;
  static constexpr uint32_t B_STAGE = KG * B_SUB;
  static constexpr uint32_t SMEM_A = 0;
  static constexpr uint32_t SMEM_B = SMEM_A + STAGES * A_STAGE;
  static constexpr uint32_t SFA_STAGE = KG * G * SF_BLOCK;      // G blocks per K block
  static constexpr uint32_t SFB_STAGE = KG * 2 * G * SF_BLOCK;  // 2 G blocks per K block
  static constexpr uint32_t SMEM_SFA = SMEM_B + STAGES * B_STAGE;
  static constexpr uint32_t SMEM_SFB = SMEM_SFA + STAGES * SFA_STAGE;
  // Scale staging for the grouped loader: per group of GROUP K blocks, one 16-byte chunk
  // (16 / CPK K blocks of codes) of each of this CTA's 128 token rows and the tile's 256
  // weight rows.
  static constexpr int KPC = 16 / CPK;  // K blocks per 16-byte chunk
  static constexpr int GROUP = KPC > KG ? KPC : KG;
  static_assert(GROUP == KPC && GROUP % KG == 0, "a chunk covers whole ring stages");
  static constexpr uint32_t STG_A = 128 * 16;
  static constexpr uint32_t STG_SLOT = STG_A + 256 * 16;
  // groups fetched ahead by a loader: 8 K blocks of 128 with one loader (4 of 256 for nvfp4's
  // one-block groups); two of its own groups with two loaders (4 groups of the walk).  Slots
  // per loader: with two, a group's slot takes the fetch STG_AHEAD groups on, issued by the
  // same lanes after they consumed it (each lane reads back only the rows it fetched)
  static constexpr int STG_AHEAD = LOADERS == 2 ? 2 : (GROUP == 1 ? 4 : 2);
  static constexpr int STG_SLOTS = LOADERS == 2 ? STG_AHEAD : STG_AHEAD + 1;
  static constexpr uint32_t SMEM_STG = SMEM_SFB + STAGES * SFB_STAGE;
  static constexpr uint32_t SMEM_CTL = SMEM_STG + LOADERS * STG_SLOTS * STG_SLOT;
  // both CTAs' bytes of one K block (the padded weight load counts the packed bytes it reads)
  static constexpr uint32_t SUB_TX = 2 * (A_SUB + (FMT_ == PF_MIXED ? B_SUB / 2 : B_SUB));
  // Row-major scale copies in flight before the oldest is announced.  A stage's copies start
  // once the MMA has freed it; announcing stage s only after the copies of s + L are issued
  // waits for the MMA to free s + L, so L <= STAGES - 2 keeps that off the MMA's path.
  static constexpr int SCALE_LOOKAHEAD = 1;
  static_assert(SCALE_LOOKAHEAD <= STAGES - 2, "scale announce would wait on the MMA");
  // scale-factor TMEM addresses on 4-column boundaries
  static_assert(PLAN.a_scale_offset % 4 == 0 && PLAN.b_scale_offset % 4 == 0 &&
                    PLAN.b_scale_offset + SF_SLOTS * SFB_COLS <= 512 &&
                    PLAN.a_scale_cols == SF_SLOTS * SFA_COLS &&
                    PLAN.b_scale_cols == SF_SLOTS * SFB_COLS,
                "scale columns of the plan");
  static_assert(PLAN.early_release_subtile < 128 / EPI_N,
                "the overlap lies in the first column half of an accumulator");
};
// the plan of the MXFP8 form, pinned to the example's values for BLOCK_K 128, VEC 32
static_assert(PCfg<PF_MXFP8>::PLAN.right_offset == 244 &&
              PCfg<PF_MXFP8>::PLAN.a_scale_offset == 500 &&
              PCfg<PF_MXFP8>::PLAN.b_scale_offset == 504 &&
              PCfg<PF_MXFP8>::PLAN.early_release_subtile == 0,
              "plan for BLOCK_K 128, VEC 32");
// the example's first worked plan (BLOCK_K 256, VEC 16); the nvfp4 form's slots are two
// such K blocks
static_assert(tmem_overlap_plan(256, EPI_N, 16, true, BN, 512).right_offset == 208 &&
              tmem_overlap_plan(256, EPI_N, 16, true, BN, 512).a_scale_offset == 464 &&
              tmem_overlap_plan(256, EPI_N, 16, true, BN, 512).b_scale_offset == 480 &&
              tmem_overlap_plan(256, EPI_N, 16, true, BN, 512).early_release_subtile == 1,
              "plan for BLOCK_K 256, VEC 16");

template <class C>
struct Ctl {
  uint64_t full[C::STAGES];
  uint64_t empty[C::STAGES];
  uint64_t sready[C::STAGES];   // SF_ST: this CTA's packed scale blocks of the stage written
  uint64_t sfull[C::SF_SLOTS];  // SF_ST: a scale slot stored by the writers of both CTAs
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t overlap;
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

__device__ __forceinline__ void record_error(int* err, int code, volatile int* abort) {
  atomicCAS(err, 0, code);
  *abort = 1;
}

__device__ __forceinline__ uint64_t sf_block_desc(uint32_t saddr) {
  return make_smem_desc(saddr, 0, 128, LAYOUT_NONE);
}

// PACKED_B: weight scales pre-packed in [E][N/128][K/128] blocks of 512 bytes (else
// row-major [E, N, K/32]); an instantiation each, so the row-major loader carries no branch.
template <int FMT, bool PACKED_B>
__global__ void __launch_bounds__(PCfg<FMT>::THREADS, 1)
bsmxfp8_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmArgs args) {
  using C = PCfg<FMT>;
  constexpr int STAGES = C::STAGES, KG = C::KG, GROUP = C::GROUP, STG_SLOTS = C::STG_SLOTS;
  constexpr int SCALE_LOOKAHEAD = C::SCALE_LOOKAHEAD;
  constexpr uint32_t A_SUB = C::A_SUB, B_SUB = C::B_SUB, A_STAGE = C::A_STAGE,
                     B_STAGE = C::B_STAGE, SFA_STAGE = C::SFA_STAGE, SFB_STAGE = C::SFB_STAGE;
  constexpr uint32_t SMEM_A = C::SMEM_A, SMEM_B = C::SMEM_B, SMEM_SFA = C::SMEM_SFA,
                     SMEM_SFB = C::SMEM_SFB, SMEM_STG = C::SMEM_STG, SMEM_CTL = C::SMEM_CTL;
  constexpr uint32_t STG_A = C::STG_A, STG_SLOT = C::STG_SLOT, SUB_TX = C::SUB_TX;
  constexpr TmemPlan PLAN = C::PLAN;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Ctl<C>* ctl = reinterpret_cast<Ctl<C>*>(smem + SMEM_CTL);
  volatile int* abort = &ctl->abort;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const int KB = args.K / C::KBLK;      // K blocks (a 128-byte operand row each)
  const int scale_row = args.K / C::VEC;  // scale codes per row
  const uint32_t rank = cluster_ctarank();
  const int64_t tile0 = blockIdx.x / 2;
  const int64_t tile_stride = gridDim.x / 2;

  // The fp4 forms take their scales through the grouped loader only (the host launches them
  // on chunkable rows: KB % GROUP == 0, scale rows of whole 16-byte chunks, aligned arrays).
  if constexpr (C::FP4) {
    if (KB % GROUP != 0 || scale_row % 16 != 0 ||
        reinterpret_cast<uintptr_t>(args.a_scales) % 16 != 0 ||
        reinterpret_cast<uintptr_t>(args.b_scales) % 16 != 0 || PACKED_B) {
      if (threadIdx.x == 0) atomicCAS(args.err, 0, DEV_TIMEOUT);
      return;
    }
  }
  if (warp == 0) {
    int status;
    int64_t row_tiles;
    validate_offsets<BM>(args.offsets, args.expert_ids, args.E, args.num_experts, args.M_total,
                            args.min_group_rows, args.max_group_rows, DEV_BAD_OFFSETS, DEV_BAD_EXPERT_IDS, status, row_tiles);
    if (lane == 0) {
      ctl->valid = status == 0;
      ctl->total_tiles = row_tiles * ((args.N + BN - 1) / BN);
      ctl->abort = 0;
      if (status && blockIdx.x == 0) atomicCAS(args.err, 0, status);
    }
  }
  __syncthreads();
  const int64_t total_tiles = ctl->total_tiles;
  if (!ctl->valid || tile0 >= total_tiles) return;

  const uint32_t sA = smem_u32(smem + SMEM_A);
  const uint32_t sB = smem_u32(smem + SMEM_B);
  const uint32_t sSFA = smem_u32(smem + SMEM_SFA);
  const uint32_t sSFB = smem_u32(smem + SMEM_SFB);
  auto full_bar = [&](int s) { return smem_u32(&ctl->full[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&ctl->empty[s]); };
  auto accf_bar = [&](int s) { return smem_u32(&ctl->acc_full[s]); };
  auto acce_bar = [&](int s) { return smem_u32(&ctl->acc_empty[s]); };
  const uint32_t ovl_bar = smem_u32(&ctl->overlap);

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    for (int s = 0; s < STAGES; ++s) {
      // leader producer (+ both CTAs' bytes) + the scale loaders of both CTAs
      mbar_init(full_bar(s), 3);  // the leader's TMA bytes + one scale loader of each CTA
      mbar_init(empty_bar(s), 1);  // one (multicast) MMA commit
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(accf_bar(s), 1);
      mbar_init(acce_bar(s), NUM_EPI_WARPS * 2);
    }
    mbar_init(ovl_bar, NUM_EPI_WARPS);  // the 4 overlap-owning warps of each CTA
    if constexpr (C::SF_ST) {
      for (int s = 0; s < STAGES; ++s) mbar_init(smem_u32(&ctl->sready[s]), 1);  // its loader
      for (int s = 0; s < C::SF_SLOTS; ++s)  // 4 writers x 2 CTAs
        mbar_init(smem_u32(&ctl->sfull[s]), 8);
    }
    mbar_init(smem_u32(&ctl->mma_done), 1);
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc<2>(smem_u32(&ctl->tmem_base), 512);
    tmem_relinquish<2>();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    // =============================== TMA producer ===============================
    if (lane == 0) {
      GroupedScheduler<BM, BN, TILE_BAND> sched;
      // The band of row strips walked together keeps its rows of A in L2 while the columns of
      // B stream past (each B column is read by the band's tiles in the same wave): A is the
      // operand to keep.
      const uint64_t pol_a = l2_policy_evict_last();
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      bool ok = true;
      TileCoord tc;
      for (int64_t t = tile0; ok && t < total_tiles; t += tile_stride) {
        if (!sched.locate(args, t, tc)) break;
        const int32_t a_row = (int32_t)(tc.m0 + 128 * rank);
        const int32_t b_row = tc.be * args.N + tc.n0 + 128 * rank;
        for (int kb0 = 0; kb0 < KB; kb0 += KG) {
          const int nk = KB - kb0 < KG ? KB - kb0 : KG;  // K blocks in this ring stage
          if (!mbar_wait(empty_bar(stage), phase ^ 1, abort)) {
            record_error(args.err, DEV_TIMEOUT, abort);
            ok = false;
            break;
          }
          const uint32_t bar = mapa_shared(full_bar(stage), 0);
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), nk * SUB_TX);
          for (int u = 0; u < nk; ++u) {
            const int kb = kb0 + u;
            tma_load_2d_pair_hint(sA + stage * A_STAGE + u * A_SUB, &tmA, kb * BK, a_row, bar,
                                  pol_a);
            tma_load_2d_pair(sB + stage * B_STAGE + u * B_SUB, &tmB, kb * BK, b_row, bar);
          }
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      const int64_t pending = issued < STAGES ? issued : STAGES;
      for (int64_t i = 0; i < pending; ++i) {
        stage = (stage + STAGES - 1) % STAGES;
        if (stage == STAGES - 1) phase ^= 1;
        mbar_wait_timed(empty_bar(stage), phase);  // consumed by the MMA -> landed
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================ MMA thread ================================
    if (lane == 0 && rank == 0) {
      GroupedScheduler<BM, BN, TILE_BAND> sched;
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      int64_t i = 0;  // tiles issued by this pair
      uint32_t sslot = 0, sphase = 0;  // SF_ST: the next K block's scale slot and its use
      TileCoord tc;
      for (int64_t t = tile0; ok && t < total_tiles; t += tile_stride, ++i) {
        if (!sched.locate(args, t, tc)) break;
        const uint32_t buf = (uint32_t)(i & 1);
        // the accumulator this tile reuses was drained (tile i-2), and the columns it shares
        // with the other accumulator were drained by tile i-1's epilogue
        if (!mbar_wait(acce_bar(buf), (uint32_t)(((i >> 1) & 1) ^ 1), abort) ||
            !mbar_wait(ovl_bar, (uint32_t)((i + 1) & 1), abort)) {
          record_error(args.err, DEV_TIMEOUT, abort);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (buf ? PLAN.right_offset : PLAN.left_offset);
        const uint32_t sfa_t = tmem_base + PLAN.a_scale_offset;
        const uint32_t sfb_t = tmem_base + PLAN.b_scale_offset;
        for (int kb0 = 0; kb0 < KB; kb0 += KG) {
          const int nk = KB - kb0 < KG ? KB - kb0 : KG;
          if (!mbar_wait(full_bar(stage), phase, abort)) {
            record_error(args.err, DEV_TIMEOUT, abort);
            ok = false;
            break;
          }
          tc_fence_after();
          for (int u = 0; u < nk; ++u) {
            uint32_t sfa_k = sfa_t, sfb_k = sfb_t;
            if constexpr (C::SF_ST) {
              // the writers of both CTAs stored this K block's scales into slot sslot
              if (!mbar_wait(smem_u32(&ctl->sfull[sslot]), sphase, abort)) {
                record_error(args.err, DEV_TIMEOUT, abort);
                ok = false;
                break;
              }
              tc_fence_after();
              sfa_k = sfa_t + sslot * C::SFA_COLS;
              sfb_k = sfb_t + sslot * C::SFB_COLS;
              if (++sslot == C::SF_SLOTS) { sslot = 0; sphase ^= 1; }
            } else {
              // this K block's scales into the TMEM scale columns (after the previous K
              // block's MMAs, which read them, in this thread's issue order); scale group g:
              // this CTA's token rows into 4 columns at sfa_t + 4g, the tile's 256 weight
              // rows into 8 columns at sfb_t + 8g (two 128-row blocks)
              const uint32_t sfa_s = sSFA + stage * SFA_STAGE + u * C::G * SF_BLOCK;
              const uint32_t sfb_s = sSFB + stage * SFB_STAGE + u * 2 * C::G * SF_BLOCK;
#pragma unroll
              for (int g = 0; g < C::G; ++g) {
                tmem_cp_32x128b_warpx4<2>(sfa_t + 4 * g, sf_block_desc(sfa_s + g * SF_BLOCK));
                tmem_cp_32x128b_warpx4<2>(sfb_t + 8 * g,
                                          sf_block_desc(sfb_s + 2 * g * SF_BLOCK));
                tmem_cp_32x128b_warpx4<2>(sfb_t + 8 * g + 4,
                                          sf_block_desc(sfb_s + (2 * g + 1) * SF_BLOCK));
              }
            }
            const uint64_t adesc = kmajor_sw128_desc(sA + stage * A_STAGE + u * A_SUB);
            const uint64_t bdesc = kmajor_sw128_desc(sB + stage * B_STAGE + u * B_SUB);
            // four MMAs per 128-byte row: K = 32 (e4m3, padded e2m1) or 64 (packed e2m1)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t acc = (kb0 + u > 0 || k > 0) ? 1u : 0u;
              const uint64_t ad = adesc + (uint64_t)(k * 2), bd = bdesc + (uint64_t)(k * 2);
              if constexpr (FMT == PF_MXFP8)
                umma_mxf8f6f4<2>(d_tmem, ad, bd, idesc_mxf8f6f4_e4m3(BM, BN, k, k), sfa_k, sfb_k,
                                 acc);
              else if constexpr (FMT == PF_MIXED)
                umma_mxf8f6f4<2>(d_tmem, ad, bd,
                                 idesc_mxf8f6f4(BM, BN, MXF_E4M3, MXF_E2M1, k, k), sfa_k, sfb_k,
                                 acc);
              else if constexpr (FMT == PF_MXF4)  // group k / 2, byte pair 2 (k % 2)
                umma_mxf4<2>(d_tmem, ad, bd, idesc_mxf4_e2m1(BM, BN, 2 * (k & 1), 2 * (k & 1)),
                             sfa_k + 4 * (k >> 1), sfb_k + 8 * (k >> 1), acc);
              else  // UE4M3 per 16: group k
                umma_mxf4nvf4_4x<2>(d_tmem, ad, bd, idesc_nvf4_e2m1_ue4m3(BM, BN),
                                    sfa_k + 4 * k, sfb_k + 8 * k, acc);
            }
          }
          if (!ok) break;
          umma_commit_pair(empty_bar(stage), 0x3);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        umma_commit_pair(accf_bar(buf), 0x3);
      }
      // every MMA issued has finished before TMEM is released; a wait that gives up is
      // reported and waited out once more (bounded) before the teardown
      umma_commit_pair(smem_u32(&ctl->mma_done), 0x1);
      if (!mbar_wait_timed(smem_u32(&ctl->mma_done), 0)) {
        record_error(args.err, DEV_TIMEOUT, abort);
        mbar_wait_timed(smem_u32(&ctl->mma_done), 0);
      }
    }
    __syncwarp();
  } else if (warp == 2 || (C::LOADERS == 2 && warp == 3)) {
    // =============================== scale loader ===============================
    // Per stage: this CTA's 128 token rows (one packed block) and all 256 weight rows of
    // the tile (two packed blocks, duplicated in both CTAs: the pair MMA reads the weight
    // scales from each CTA's own TMEM).  Announced on the MMA CTA's full barrier.
    const uint8_t* a_sc = static_cast<const uint8_t*>(args.a_scales);
    const uint8_t* b_sc = static_cast<const uint8_t*>(args.b_scales);
    // weight scales either row-major [E, N, K/32] or pre-packed [E][N/128][K/128] blocks
    constexpr bool packed_b = PACKED_B;
    const bool second = C::LOADERS == 2 && warp == 3;
    const int nblk = args.N / 128;
    GroupedScheduler<BM, BN, TILE_BAND> sched;
    uint32_t stage = 0, phase = 0;
    // Grouped path: when a row's codes for GROUP consecutive K blocks form one aligned
    // 16-byte chunk (scale rows of whole chunks, 16-byte aligned scale arrays), fetch a group
    // per row with one 16-byte copy, STG_AHEAD groups ahead, and transpose each K block's
    // words into its packed blocks (one per scale group) in shared memory.
    const bool grouped = (KB % GROUP == 0) && (scale_row % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(a_sc) % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(b_sc) % 16 == 0);
    if (grouped) {
      // Two loaders: the walk's groups alternate between them (group g to warp 2 + g % 2),
      // each loader with its own staging slots.
      const int NG = KB / GROUP;  // groups per tile
      const uint32_t stg_off = second ? STG_SLOTS * STG_SLOT : 0;
      const uint32_t sSTG = smem_u32(smem + SMEM_STG) + stg_off;
      const uint8_t* stg = smem + SMEM_STG + stg_off;
      GroupedScheduler<BM, BN, TILE_BAND> pre;
      TileCoord tp;
      int64_t tp_t = tile0;
      bool pre_ok = pre.locate(args, tp_t, tp);
      int qp = 0;
      auto next_pre = [&]() {  // the walk's next group
        if (pre_ok && ++qp == NG) {
          qp = 0;
          tp_t += tile_stride;
          pre_ok = tp_t < total_tiles && pre.locate(args, tp_t, tp);
        }
      };
      if (second) next_pre();
      auto issue_group = [&](int slot) {
        if (pre_ok) {
          const uint32_t dst = sSTG + slot * STG_SLOT;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = 32 * i + (int)lane;
            const int64_t m = tp.m0 + 128 * rank + r;
            const bool live = m < args.M_total;
            cp_async_16(dst + r * 16, live ? a_sc + m * scale_row + 16 * qp : a_sc, live ? 16u : 0u);
          }
          if constexpr (packed_b) {
            // pre-packed weight scales: the tile's two 128-row blocks of these 4 K blocks are
            // two contiguous 2 KB runs (staging: [block h][K block][512 bytes])
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int nb = tp.n0 / 128 + h;
              const bool live = nb < nblk;
              const uint8_t* run = b_sc + (((int64_t)tp.be * nblk + nb) * KB + 4 * qp) * SF_BLOCK;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int c = 32 * i + (int)lane;
                cp_async_16(dst + STG_A + h * 4 * SF_BLOCK + c * 16, live ? run + c * 16 : b_sc,
                            live ? 16u : 0u);
              }
            }
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int r = 32 * i + (int)lane;  // weight rows 32i + lane
              const int n = tp.n0 + r;
              const bool live = n < args.N;
              const uint8_t* src = b_sc + ((int64_t)tp.be * args.N + n) * scale_row + 16 * qp;
              cp_async_16(dst + STG_A + r * 16, live ? src : b_sc, live ? 16u : 0u);
            }
          }
        }
        for (int l = 0; l < C::LOADERS; ++l) next_pre();
        cp_async_commit();  // an empty group keeps the group count in step
      };
      for (int a = 0; a < C::STG_AHEAD; ++a) issue_group(a);
      int64_t g = 0;   // groups of the walk
      int64_t og = 0;  // this loader's groups
      bool ok = true;
      TileCoord tc;
      for (int64_t t = tile0; ok && t < total_tiles; t += tile_stride) {
        if (!sched.locate(args, t, tc)) break;
        for (int q = 0; ok && q < NG; ++q, ++g) {
          if (C::LOADERS == 2 && (int)(g & 1) != (int)second) {  // the other loader's group
            for (int jg = 0; jg < GROUP; jg += KG)
              if (++stage == STAGES) { stage = 0; phase ^= 1; }
            continue;
          }
          cp_async_wait_group<C::STG_AHEAD - 1>();  // group og has landed (later in flight)
          __syncwarp();
          const uint8_t* src = stg + (og % STG_SLOTS) * STG_SLOT;
          for (int jg = 0; jg < GROUP; jg += KG) {
            const bool got =
                __all_sync(0xffffffffu, mbar_wait(empty_bar(stage), phase ^ 1, abort));
            if (!got) {
              if (lane == 0) record_error(args.err, DEV_TIMEOUT, abort);
              ok = false;
              break;
            }
#pragma unroll
            for (int u = 0; u < KG; ++u) {
            const int j = jg + u;
            // 128 rows (row 32*rg + lane at staging byte (32*rg + lane)*16) into the G packed
            // blocks of K block j, block b (codes 4b..4b+3) at dst + b * step: each lane loads
            // its 4 rows' CPK codes of the K block (one 4-, 8- or 16-byte load per row) and
            // writes row 32*rg + lane's word of group b at byte lane*16 + rg*4
            auto transpose = [&](const uint8_t* rows, uint8_t* dst, uint32_t step) {
              uint32_t w[4][C::G];
#pragma unroll
              for (int rg = 0; rg < 4; ++rg) {
                const uint8_t* r = rows + (32 * rg + lane) * 16 + C::CPK * j;
                if constexpr (C::G == 4) {
                  const uint4 v = *reinterpret_cast<const uint4*>(r);
                  w[rg][0] = v.x; w[rg][C::G > 1 ? 1 : 0] = v.y;
                  w[rg][C::G > 2 ? 2 : 0] = v.z; w[rg][C::G > 3 ? 3 : 0] = v.w;
                } else if constexpr (C::G == 2) {
                  const uint2 v = *reinterpret_cast<const uint2*>(r);
                  w[rg][0] = v.x; w[rg][C::G > 1 ? 1 : 0] = v.y;
                } else {
                  w[rg][0] = *reinterpret_cast<const uint32_t*>(r);
                }
              }
#pragma unroll
              for (int b = 0; b < C::G; ++b)
                *reinterpret_cast<uint4*>(dst + b * step + lane * 16) =
                    make_uint4(w[0][b], w[1][b], w[2][b], w[3][b]);
            };
            uint8_t* sfa = smem + SMEM_SFA + stage * SFA_STAGE + u * C::G * SF_BLOCK;
            uint8_t* sfb = smem + SMEM_SFB + stage * SFB_STAGE + u * C::G * 2 * SF_BLOCK;
            if constexpr (packed_b) {  // (MX-coded forms: one group, one loader)
              transpose(src, sfa, SF_BLOCK);
              const uint8_t* pb = src + STG_A + j * SF_BLOCK + lane * 16;
              reinterpret_cast<uint4*>(sfb)[lane] = *reinterpret_cast<const uint4*>(pb);
              reinterpret_cast<uint4*>(sfb)[32 + lane] =
                  *reinterpret_cast<const uint4*>(pb + 4 * SF_BLOCK);
            } else {
              transpose(src, sfa, SF_BLOCK);
              transpose(src + STG_A, sfb, 2 * SF_BLOCK);                    // weight rows 0-127
              transpose(src + STG_A + 128 * 16, sfb + SF_BLOCK, 2 * SF_BLOCK);  // 128-255
            }
            }
            fence_proxy_async_smem();  // generic-proxy writes -> tcgen05.cp (async proxy)
            __syncwarp();
            if (lane == 0) {
              mbar_arrive_cluster(mapa_shared(full_bar(stage), 0));
              if constexpr (C::SF_ST) mbar_arrive(smem_u32(&ctl->sready[stage]));
            }
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          __syncwarp();
          // one loader: group og - 1's slot is free; two: this group's own slot
          issue_group((int)((og + C::STG_AHEAD) % STG_SLOTS));
          ++og;
        }
      }
      cp_async_wait_group<0>();
    } else if constexpr (!C::FP4) {
    // (the fp4 forms never get here: the kernel winds down at its start on such rows)
    uint32_t ring[SCALE_LOOKAHEAD + 1] = {};
    int inflight = 0, head = 0;
    bool ok = true;
    TileCoord tc;
    auto announce_oldest = [&]() {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(full_bar(ring[head]), 0));
      head = (head + 1) % (SCALE_LOOKAHEAD + 1);
      --inflight;
    };
    for (int64_t t = tile0; ok && t < total_tiles; t += tile_stride) {
      if (!sched.locate(args, t, tc)) break;
      for (int kb0 = 0; kb0 < KB; kb0 += KG) {
        const int nk = KB - kb0 < KG ? KB - kb0 : KG;
        const bool got = __all_sync(0xffffffffu, mbar_wait(empty_bar(stage), phase ^ 1, abort));
        if (!got) {
          if (lane == 0) record_error(args.err, DEV_TIMEOUT, abort);
          ok = false;
          break;
        }
        for (int u = 0; u < nk; ++u) {
        const int kb = kb0 + u;
        const uint32_t da = sSFA + stage * SFA_STAGE + u * SF_BLOCK + lane * 16;
        const uint32_t db = sSFB + stage * SFB_STAGE + u * 2 * SF_BLOCK + lane * 16;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = j * 32 + (int)lane;
          const int64_t m = tc.m0 + 128 * rank + r;
          const bool a_live = m < args.M_total;
          cp_async_4(da + 4 * j, a_live ? a_sc + m * scale_row + 4 * kb : a_sc, a_live ? 4u : 0u);
          if constexpr (!packed_b) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int n = tc.n0 + 128 * h + r;
              const bool b_live = n < args.N;
              const uint8_t* src = b_sc + ((int64_t)tc.be * args.N + n) * scale_row + 4 * kb;
              cp_async_4(db + h * SF_BLOCK + 4 * j, b_live ? src : b_sc, b_live ? 4u : 0u);
            }
          }
        }
        if constexpr (packed_b) {
          // pre-packed weight scales: the stage's two blocks, 16 bytes per lane each
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int nb = tc.n0 / 128 + h;
            const bool live = nb < nblk;
            const uint8_t* blk = b_sc + (((int64_t)tc.be * nblk + nb) * KB + kb) * SF_BLOCK;
            cp_async_16(db + h * SF_BLOCK, live ? blk + lane * 16 : b_sc, live ? 16u : 0u);
          }
        }
        }
        cp_async_commit();
        ring[(head + inflight) % (SCALE_LOOKAHEAD + 1)] = stage;
        ++inflight;
        if (inflight > SCALE_LOOKAHEAD) {
          cp_async_wait_group<SCALE_LOOKAHEAD>();
          announce_oldest();
        }
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
    cp_async_wait_group<0>();
    while (inflight > 0) announce_oldest();
    }
  } else if (C::SF_ST && warp >= EPI_WARP0 + NUM_EPI_WARPS) {
    // ============================== scale writers ===============================
    // Warp 12 + q stores TMEM lane quarter q of K block i's scale slot (i % SF_SLOTS) from
    // this CTA's packed blocks of the stage: for the token rows (the MMA's M operand) only
    // column q of each 4-column group is read, row 32q + r's codes at lane r; for the tile's
    // 256 weight rows (its N operand) every lane quarter reads row 32j + r at lane r of column
    // j (j < 8).  A slot is stored again only after the MMAs that read it, SF_SLOTS K blocks
    // earlier, completed (the commit on that K block's stage).
    static_assert(!C::SF_ST || (KG == 1 && C::SF_SLOTS < STAGES),
                  "one K block per ring stage; a slot's reuse is within the ring");
    const uint32_t q = warp & 3;
    GroupedScheduler<BM, BN, TILE_BAND> sched;
    uint32_t stage = 0, phase = 0;
    uint32_t slot = 0;
    int64_t kbi = 0;  // K blocks stored by this warp
    bool ok = true;
    TileCoord tc;
    for (int64_t t = tile0; ok && t < total_tiles; t += tile_stride) {
      if (!sched.locate(args, t, tc)) break;
      for (int kb = 0; kb < KB; ++kb, ++kbi) {
        bool got = mbar_wait(smem_u32(&ctl->sready[stage]), phase, abort);
        if (got && kbi >= C::SF_SLOTS) {
          // K block j = kbi - SF_SLOTS (same slot): the commit of its stage, its use j / STAGES
          const int64_t j = kbi - C::SF_SLOTS;
          got = mbar_wait(empty_bar((int)(j % STAGES)), (uint32_t)((j / STAGES) & 1), abort);
        }
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) record_error(args.err, DEV_TIMEOUT, abort);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t lanes = (q * 32) << 16;
        const uint32_t ta = tmem_base + lanes + PLAN.a_scale_offset + slot * C::SFA_COLS;
        const uint32_t tb = tmem_base + lanes + PLAN.b_scale_offset + slot * C::SFB_COLS;
#pragma unroll
        for (int g = 0; g < C::G; ++g) {
          // a packed block holds row 32c + r's 4 codes at byte 16r + 4c
          const uint8_t* pa = smem + SMEM_SFA + stage * SFA_STAGE + g * SF_BLOCK + lane * 16;
          tmem_st_32x32b_x1(ta + 4 * g + q, *reinterpret_cast<const uint32_t*>(pa + 4 * q));
          const uint8_t* pb = smem + SMEM_SFB + stage * SFB_STAGE + 2 * g * SF_BLOCK + lane * 16;
          const uint4 lo = *reinterpret_cast<const uint4*>(pb);
          const uint4 hi = *reinterpret_cast<const uint4*>(pb + SF_BLOCK);
          const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
          tmem_st_32x32b_x8(tb + 8 * g, w);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->sfull[slot]), 0));
        if (++slot == C::SF_SLOTS) slot = 0;
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
  } else if (warp >= EPI_WARP0 && warp < EPI_WARP0 + NUM_EPI_WARPS) {
    // ================================= epilogue =================================
    const uint32_t ew = warp - EPI_WARP0;
    const uint32_t quarter = warp & 3;
    const uint32_t half = ew >> 2;  // accumulator columns half*128 .. +127
    __nv_bfloat16* Cmat = static_cast<__nv_bfloat16*>(args.C);
    GroupedScheduler<BM, BN, TILE_BAND> sched;
    const uint64_t pol_c = l2_policy_evict_first();
    // a 32-byte aligned C takes one full L2 sector per 32-byte store
    const bool c_vec32 = (reinterpret_cast<uintptr_t>(args.C) & 31) == 0;
    int64_t i = 0;
    TileCoord tc;
    for (int64_t t = tile0; t < total_tiles; t += tile_stride, ++i) {
      if (!sched.locate(args, t, tc)) break;
      const uint32_t buf = (uint32_t)(i & 1);
      const bool got =
          __all_sync(0xffffffffu, mbar_wait(accf_bar(buf), (uint32_t)((i >> 1) & 1), abort));
      if (!got) {
        if (lane == 0) record_error(args.err, DEV_TIMEOUT, abort);
        break;
      }
      tc_fence_after();
      const uint32_t col_base = buf ? PLAN.right_offset : PLAN.left_offset;
      // even tiles drain high -> low, odd tiles low -> high: the shared columns come first
      const bool high_first = (buf == 0);
      const bool owns_overlap = high_first ? (half == 1) : (half == 0);
      const int64_t row = tc.m0 + 128 * rank + quarter * 32 + lane;
      const uint32_t taddr = tmem_base + ((quarter * 32) << 16) + col_base;
      // drain step s: subtile high_first ? 3 - s : s of this warp's column half
      auto col_of = [&](int s) { return (int)half * 128 + (high_first ? 3 - s : s) * EPI_N; };
      auto load_bf16 = [&](int s, uint32_t (&p)[16]) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + col_of(s), v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          p[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
      };
      auto store_bf16 = [&](int s, const uint32_t (&p)[16]) {
        const int n = tc.n0 + col_of(s);
        if (row < tc.m_end && n < args.N) {
          __nv_bfloat16* dst = Cmat + row * (int64_t)args.N + n;
          if (c_vec32) {  // N % 128 == 0: dst is 32-byte aligned when C is
            const uint32_t lo[8] = {p[0], p[1], p[2], p[3], p[4], p[5], p[6], p[7]};
            const uint32_t hi[8] = {p[8], p[9], p[10], p[11], p[12], p[13], p[14], p[15]};
            st_global_v8_hint(dst, lo, pol_c);
            st_global_v8_hint(dst + 16, hi, pol_c);
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_global_v4_hint(dst + 8 * q, p[4 * q], p[4 * q + 1], p[4 * q + 2],
                                p[4 * q + 3], pol_c);
          }
        }
      };
      // The warps owning the shared columns read every subtile up to the plan's release
      // point out of TMEM before storing any of them: the next tile's MMAs wait on that
      // release, and a lane's 16-byte stores to its own row of C (32 rows per instruction)
      // hold the warp for hundreds of cycles per subtile.
      constexpr int E = PLAN.early_release_subtile;
      int s0 = 0;
      if (owns_overlap) {
        uint32_t head[E + 1][16];
#pragma unroll
        for (int s = 0; s <= E; ++s) load_bf16(s, head[s]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(ovl_bar, 0));
#pragma unroll
        for (int s = 0; s <= E; ++s) store_bf16(s, head[s]);
        s0 = E + 1;
      }
      for (int s = s0; s < 4; ++s) {
        uint32_t p[16];
        load_bf16(s, p);
        store_bf16(s, p);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(buf), 0));
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<2>(tmem_base, 512);
  }
}

}  // namespace mxp

namespace mxp {
template <int FMT, bool PACKED_B>
cudaError_t launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& args,
                   int num_sms, cudaStream_t stream) {
  using C = PCfg<FMT>;
  static_assert(smem_bytes<C>() <= 232448, "shared memory budget");
  static std::atomic<bool> attr_set[64];  // per device; several host threads may launch
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(bsmxfp8_pair_kernel<FMT, PACKED_B>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes<C>());
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set[dev].store(true, std::memory_order_release);
  }
  const int64_t max_row_tiles = (args.M_total + mxp::BM - 1) / mxp::BM + args.E;
  const int64_t max_tiles = max_row_tiles * ((args.N + mxp::BN - 1) / mxp::BN);
  const int64_t pairs = num_sms / 2;
  const int grid = (int)((max_tiles < pairs ? max_tiles : pairs) * 2);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = smem_bytes<C>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bsmxfp8_pair_kernel<FMT, PACKED_B>, tmA, tmB, args);
}
}  // namespace mxp

cudaError_t launch_bsmxfp8_pair(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                const GemmArgs& args, int num_sms, cudaStream_t stream) {
  return args.b_scales_packed ? mxp::launch<mxp::PF_MXFP8, true>(tmA, tmB, args, num_sms, stream)
                              : mxp::launch<mxp::PF_MXFP8, false>(tmA, tmB, args, num_sms, stream);
}

cudaError_t launch_bsmx_pair_fp4(int fmt, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                 const GemmArgs& args, int num_sms, cudaStream_t stream) {
  using namespace mxp;
  switch (fmt) {
    case PF_MIXED:
      return args.b_scales_packed ? launch<PF_MIXED, true>(tmA, tmB, args, num_sms, stream)
                                  : launch<PF_MIXED, false>(tmA, tmB, args, num_sms, stream);
    case PF_MXF4: return launch<PF_MXF4, false>(tmA, tmB, args, num_sms, stream);
    case PF_NVF4: return launch<PF_NVF4, false>(tmA, tmB, args, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

TmemPlan mx_pair_tmem_plan() { return mxp::PCfg<mxp::PF_MXFP8>::PLAN; }

}  // namespace bsfp8

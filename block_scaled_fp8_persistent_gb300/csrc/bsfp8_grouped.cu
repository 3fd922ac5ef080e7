// Blockwise-scaled FP8 grouped GEMM for sm_103a (persistent, warp specialized).
//
//   C[m, n] = sum_kb a_scales[kb, m] * b_scales[e, n/128, kb] * sum_{k in kb} A[m,k] B[e,n,k]
//
// with e the expert owning row m, 1x128 A scales and 128x128 B scales over K blocks of
// 128, fp32 accumulation and bf16 output.
//
// Prior art followed (and where this differs):
//  * promote_accumulators (MAX kernels, grouped_matmul_sm100_blockwise_fp8): every K block
//    produces a TMEM partial that the epilogue warps multiply by a_scale x b_scale and add
//    into fp32 register tiles; the B scale is read from global memory.
//  * EpilogueWarpContext.per_k_stage (MAX sm100_structured): the epilogue consumes one
//    TMEM stage per K iteration and signals the MMA warp when it is free.
//  * Triton Gluon example "Overlapping Accumulator Block-Scaled Matrix Multiplication":
//    load / MMA / epilogue partitions, persistent static tile stride, 2-CTA tiles.
//
// Roles with 96 A rows per CTA (8 warps, the layouts the planner picks).  The M = 128 MMA
// computes TMEM lanes 96..127 from shared-memory rows that nobody reads.  A warp can only
// read the TMEM lanes of its own SM sub-partition (lanes 32*(w%4)..), so the sub-partition
// of lanes 96..127 is free for the roles:
//   warp 3       TMA producer: per K block, A rows [rows x 128] and this CTA's share of B
//                rows [BN/CG x 128] (e4m3, 128-byte swizzle) into a STAGES-deep ring.
//   warp 7       TMEM owner; in the MMA CTA (rank 0 of a pair) the single issuing thread: per
//                K block 4 x tcgen05.mma kind::f8f6f4 (K = 32 each) into a fresh TMEM partial
//                (ACC_STAGES-deep ring of BN columns), then one commit to the stage's empty
//                barrier, which both the producer and the epilogue wait on.
//   warps 0-2,   epilogue: warp w reads TMEM lanes 32*(w%4).. (rows) and columns
//   4-6          (BN/2)*(w/4).. ; per K block it loads its partial, hands the TMEM stage back
//                and promotes acc = fma(sa*sb, partial, acc) in registers.  After the last K
//                block it rounds to bf16 and stores the rows of the tile's expert.
// A sub-partition that issues TMA loads or tcgen05.mma next to epilogue warps slows those
// warps down about twofold (clock64 traces: every step of their K-block loop, not one wait),
// so no epilogue warp shares a sub-partition with a role; a quarter of each single-CTA MMA
// is the price.  The 128-row single-CTA layouts (12 warps: warps 0-3 each own one operand
// stage, load it and issue its MMAs; warps 4-11 epilogue) stay selectable and parity-tested
// but run ~1.4x slower per tile.
//
// CG = 2 runs a CTA pair (cluster of 2) with the pair MMA (M = 256): each CTA's TMEM holds
// its 128 rows x BN columns; B is split between the CTAs; the TMA completions of both CTAs
// are counted on the leader's barrier and the leader's commits arrive on both CTAs'
// barriers.  Each CTA promotes and stores its own rows.  Symmetric pairs run the 96-row
// layout in both CTAs (192-row tiles).  The asymmetric pair (PEER_ROWS = 128) uses all 128
// MMA rows of the peer: the leader keeps the 96-row layout and its producer also loads the
// peer's A rows and half of B, by TMA multicast to the peer alone with the bytes counted on
// the leader's barrier, so the peer runs epilogue warps only (224-row tiles, 87.5 % of the
// MMA rows useful).
//
// A and B scales reach the epilogue through the read-only cache two K blocks ahead of their
// use, and the A scales' lines are prefetched into L1 SCALE_LOOKAHEAD K blocks ahead.
// a_scales is [K/128, M_total], so every K block touches a new line per 32 rows; loads issued
// one K block ahead, or without the L1 prefetch, left the epilogue warps waiting on them.
// With 256-column tiles each epilogue warp's 128 columns lie in one 128-column B-scale block,
// so it needs one B scale per K block (and the registers of a second one go to the loads
// in flight).
#include <atomic>
#include <cuda_bf16.h>
#include "common.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace bsfp8 {
namespace bw {

constexpr int BK = 128;
constexpr uint32_t TMEM_COLS = 512;

template <int CG_, int BN_, int STAGES_, int ACC_STAGES_, int ROWS_ = 128, int PEER_ROWS_ = ROWS_>
struct Cfg {
  static constexpr int CG = CG_;                  // CTAs per tile (1 or 2)
  static constexpr int BN = BN_;                  // tile columns
  static constexpr int ROWS = ROWS_;              // A rows per CTA (128, or 96: see above)
  // Asymmetric pair: a 96-row leader whose spare sub-partition hosts the producer and the
  // MMA issuer, and a 128-row peer that runs epilogue warps only; the leader's producer
  // loads the peer's operands (multicast to the peer alone, bytes counted on the leader).
  static constexpr int PEER_ROWS = PEER_ROWS_;    // A rows of the pair's second CTA
  static constexpr bool ASYM = CG_ == 2 && PEER_ROWS_ != ROWS_;
  static constexpr int BM = CG == 2 ? ROWS + PEER_ROWS : ROWS;  // tile rows
  static constexpr bool SPARE_QUARTER = ROWS == 96;  // TMEM lanes 96..127 unused
  static constexpr int THREADS = SPARE_QUARTER ? 256 : 384;
  static constexpr int PRODUCER_WARP = SPARE_QUARTER ? 3 : 0;
  static constexpr int MMA_WARP = SPARE_QUARTER ? 7 : 1;  // also allocates TMEM
  static constexpr int NUM_EPI_WARPS = SPARE_QUARTER ? 6 : 8;  // (the leader's, with ASYM)
  static constexpr int PAIR_EPI_WARPS = ASYM ? NUM_EPI_WARPS + 8 : NUM_EPI_WARPS * CG;
  static constexpr int STAGES = STAGES_;          // SMEM ring depth
  static constexpr int ACC_STAGES = ACC_STAGES_;  // TMEM partial ring depth
  static constexpr int B_ROWS = BN / CG;          // B rows loaded by each CTA
  static constexpr int COLS = BN / 2;             // columns per epilogue warp
  static constexpr int CHUNKS = COLS / 16;        // 16-column chunks per warp
  // all of a warp's columns fit in registers next to its accumulators: load them all,
  // release the TMEM stage, then promote
  static constexpr bool LOAD_ALL = COLS <= 96;
  // The MMA reads 128 A rows per CTA.  A one-CTA 96-row tile keeps only its 96 rows per
  // stage: rows 96..127 of the read come from the next 4 KB of shared memory (the next stage,
  // or the first B stage), land in TMEM lanes 96..127 and are never read, and the ring gets
  // a fifth stage in the same space.
  static constexpr uint32_t A_STAGE = (SPARE_QUARTER && CG == 1 ? 96 : 128) * BK;
  static constexpr uint32_t B_STAGE = B_ROWS * BK;
  static constexpr int A_BOX = ASYM ? 128 : ROWS;  // A rows per TMA box
  static constexpr uint32_t STAGE_TX = (A_BOX * BK + B_STAGE) * CG;  // bytes loaded, pair
  // each epilogue warp's columns lie in one 128-column B-scale block (one B scale per K
  // block): its first column is a multiple of COLS, which divides 128
  static constexpr bool ONE_BLOCK = 128 % COLS == 0;
  static constexpr int SCALE_LOOKAHEAD = 6;  // K blocks of A-scale L1 prefetch
  static constexpr uint32_t SMEM_A = 0;
  static constexpr uint32_t SMEM_B = SMEM_A + STAGES * A_STAGE;
  static constexpr uint32_t SMEM_CTL = SMEM_B + STAGES * B_STAGE;
  static constexpr uint32_t IDESC = idesc_f8f6f4_e4m3(128 * CG, BN);
  // Tile walk: CTA pairs take bands of 16 row tiles (row index fastest inside a band) and keep
  // the band's A rows in L2 while B streams; one-CTA tiles take the plain order (column index
  // fastest) and keep B, which the row tiles of an expert share within a wave.
  static constexpr int TILE_BAND = CG == 2 ? 16 : 1;
  static_assert(ROWS == 128 || ROWS == 96, "A rows per CTA");
  static_assert(!ASYM || (ROWS == 96 && PEER_ROWS == 128), "asymmetric pair: 96 + 128 rows");
  __device__ static bool is_epilogue(uint32_t warp) {
    return SPARE_QUARTER ? (warp & 3) != 3 : warp >= 4;
  }
  __device__ static uint32_t column_half(uint32_t warp) {
    return SPARE_QUARTER ? warp >> 2 : (warp - 4) >> 2;
  }
  // One CTA with 128 rows: every sub-partition hosts two epilogue warps, so the producer and
  // MMA work is split four ways instead of sitting on one of them: warp j of warpgroup 0
  // owns operand stage j (K blocks kb with kb % 4 == j), loads it and issues its MMAs.
  static constexpr bool ROLE4 = !SPARE_QUARTER && CG == 1;
  // TMEM-stage release barriers: one per K block mod 4 with ROLE4 (each has a single waiter,
  // which sees its phases in order), else one per TMEM stage
  static constexpr int N_TEMPTY = ROLE4 ? 4 : ACC_STAGES;
  static_assert(!ROLE4 || (STAGES == 4 && ACC_STAGES <= 4 && 4 % ACC_STAGES == 0),
                "four role warps own one operand stage each");
  static_assert(ACC_STAGES * BN <= (int)TMEM_COLS, "TMEM ring too large");
  static_assert(COLS % 16 == 0 && BN % 16 == 0 && B_ROWS % 8 == 0, "tile shape");
  static_assert(LOAD_ALL || COLS % 64 == 0, "two-phase epilogue works in 64-column halves");
  static_assert(B_STAGE % 1024 == 0, "128-byte-swizzle atoms need 1024-byte stages");
};

template <class C>
struct Ctl {
  uint64_t full[C::STAGES];
  uint64_t empty[C::STAGES];
  uint64_t tempty[C::N_TEMPTY];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  int valid;
  int pad;
  long long total_tiles;
};

template <class C>
constexpr uint32_t smem_bytes() {
  return C::SMEM_CTL + sizeof(Ctl<C>) + 1024;  // + alignment slack
}

__device__ __forceinline__ void record_error(int* err, int code, volatile int* abort) {
  atomicCAS(err, 0, code);
  *abort = 1;
}

// Promote 16 columns: acc[j] = fma(s, partial[j], acc[j]), two columns per packed fp32
// FMA (each lane of it rounds exactly like fmaf).
__device__ __forceinline__ void promote16(float2* acc, const uint32_t* p, float s) {
  const float2 s2 = make_float2(s, s);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    acc[j] = __ffma2_rn(s2, make_float2(__uint_as_float(p[2 * j]), __uint_as_float(p[2 * j + 1])),
                        acc[j]);
}

// Issue the MMAs of one K block: 4 x tcgen05.mma kind::f8f6f4 (K = 32 e4m3 each, 32 bytes
// along the swizzled row; the descriptors advance by 32 bytes >> 4) from an operand stage
// into the TMEM partial at d_tmem, then one commit to the stage's empty barrier.  That
// barrier completes when the K block's MMAs have finished: the producer waits on it to
// refill the stage and the epilogue to read the partial.
template <class C>
__device__ __forceinline__ void issue_kblock(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t empty_bar) {
#pragma unroll
  for (int k = 0; k < BK / 32; ++k)
    umma_f8f6f4<C::CG>(d_tmem, adesc + (uint64_t)(k * 2), bdesc + (uint64_t)(k * 2), C::IDESC,
                       k > 0 ? 1u : 0u);
  if constexpr (C::CG == 1) umma_commit(empty_bar);
  else umma_commit_pair(empty_bar, 0x3);
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
bsfp8_blockwise_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB, const GemmArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Ctl<C>* ctl = reinterpret_cast<Ctl<C>*>(smem + C::SMEM_CTL);
  volatile int* abort = &ctl->abort;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const int KB = args.K / BK;
  const uint32_t rank = (C::CG == 2) ? cluster_ctarank() : 0;  // 0 = MMA CTA of the pair
  const int64_t tile0 = blockIdx.x / C::CG;                    // this pair's first tile
  const int64_t tile_stride = gridDim.x / C::CG;

  // ---- work discovery: validate the offsets, count tiles (same answer in every CTA) ----
  if (warp == 0) {
    int status;
    int64_t row_tiles;
    validate_offsets<C::BM>(args.offsets, args.expert_ids, args.E, args.num_experts, args.M_total,
                            args.min_group_rows, args.max_group_rows, DEV_BAD_OFFSETS, DEV_BAD_EXPERT_IDS, status, row_tiles);
    if (lane == 0) {
      ctl->valid = status == 0;
      ctl->total_tiles = row_tiles * ((args.N + C::BN - 1) / C::BN);
      ctl->abort = 0;
      if (status && blockIdx.x == 0) atomicCAS(args.err, 0, status);
    }
  }
  __syncthreads();
  const int64_t total_tiles = ctl->total_tiles;
  if (!ctl->valid || tile0 >= total_tiles) return;  // both CTAs of a pair agree

  // ---- setup: barriers, TMEM ---------------------------------------------------------
  const uint32_t sA = smem_u32(smem + C::SMEM_A);
  const uint32_t sB = smem_u32(smem + C::SMEM_B);
  auto full_bar = [&](int s) { return smem_u32(&ctl->full[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&ctl->empty[s]); };
  auto tempty_bar = [&](int s) { return smem_u32(&ctl->tempty[s]); };

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);   // the leader's producer arrives (+ both CTAs' bytes)
      mbar_init(empty_bar(s), 1);  // one MMA commit per K block
    }
    for (int s = 0; s < C::N_TEMPTY; ++s) {
      mbar_init(tempty_bar(s), C::PAIR_EPI_WARPS);  // every epilogue warp of the pair
    }
    mbar_init(smem_u32(&ctl->mma_done), 1);
    fence_mbarrier_init();
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc<C::CG>(smem_u32(&ctl->tmem_base), TMEM_COLS);
    tmem_relinquish<C::CG>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (C::CG == 2) cluster_sync();  // peer barriers initialised before any use
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  // the asymmetric pair's peer runs epilogue warps only
  const bool all_epilogue = C::ASYM && rank == 1;
  if (!all_epilogue && !C::is_epilogue(warp)) {
    // 128 rows: warpgroup 0 (producer, MMA issuer, two idle warps) gives registers away
    if constexpr (!C::SPARE_QUARTER) asm volatile("setmaxnreg.dec.sync.aligned.u32 40;");
    if (C::ROLE4 && lane == 0) {
      // ======================= stage owner j = warp (0..3) =======================
      // K blocks g = j, j + 4, ... (counted over this CTA's tiles): wait for the stage's
      // previous MMAs, load A and B into it, wait for the bytes, wait for the TMEM stage
      // (the epilogue's release of K block g - ACC_STAGES), issue 4 MMAs, commit to the
      // stage's empty barrier.  Waits sleep (suspend-time hint): the sub-partition is shared
      // with two epilogue warps.
      const uint32_t j = warp;
      GroupedScheduler<C::BM, C::BN, C::TILE_BAND> sched;
      const uint64_t pol_b = l2_policy_evict_last();
      const uint64_t adesc = kmajor_sw128_desc(sA + j * C::A_STAGE);
      const uint64_t bdesc = kmajor_sw128_desc(sB + j * C::B_STAGE);
      int64_t g = 0;
      uint32_t u = 0;  // uses of stage j so far
      bool ok = true;
      TileCoord tc;
      for (int64_t t = tile0; ok && t < total_tiles; t += tile_stride) {
        if (!sched.locate(args, t, tc)) break;
        const int32_t a_row = (int32_t)tc.m0;
        const int32_t b_row = tc.be * args.N + tc.n0;
        // this tile's K blocks with g % 4 == j
        for (int kb = (int)((j - (uint32_t)(g & 3)) & 3); kb < KB; kb += 4) {
          const int64_t gk = g + kb;
          bool w = mbar_wait_sleep(empty_bar(j), (u & 1) ^ 1, abort);
          if (w) {
            mbar_arrive_expect_tx(full_bar(j), C::STAGE_TX);
            tma_load_2d(sA + j * C::A_STAGE, &tmA, kb * BK, a_row, full_bar(j));
            tma_load_2d_hint(sB + j * C::B_STAGE, &tmB, kb * BK, b_row, full_bar(j), pol_b);
            w = mbar_wait_sleep(full_bar(j), u & 1, abort);
          }
          const int64_t gr = gk - C::ACC_STAGES;  // its TMEM stage's previous K block
          if (w && gr >= 0) w = mbar_wait_sleep(tempty_bar((int)(gr & 3)), (uint32_t)(gr >> 2) & 1, abort);
          if (!w) {
            record_error(args.err, DEV_TIMEOUT, abort);
            ok = false;
            break;
          }
          tc_fence_after();
          issue_kblock<C>(tmem_base + (uint32_t)(gk % C::ACC_STAGES) * C::BN, adesc, bdesc,
                          empty_bar(j));
          ++u;
        }
        g += KB;
      }
      // the stage's last MMAs have finished before TMEM is released (bounded, reported)
      if (u > 0 && !mbar_wait_timed(empty_bar(j), (u - 1) & 1)) {
        record_error(args.err, DEV_TIMEOUT, abort);
        mbar_wait_timed(empty_bar(j), (u - 1) & 1);
      }
    } else if (!C::ROLE4 && warp == C::PRODUCER_WARP && lane == 0) {
      // =============================== TMA producer ===============================
      // The producer sleeps in its barrier waits (suspend-time hint): it shares its
      // sub-partition with the MMA thread, whose issue slots set the pace.
      GroupedScheduler<C::BM, C::BN, C::TILE_BAND> sched;
      // One-CTA tiles: B (expert weights) is re-read by every row tile of its expert,
      // possibly in a later wave of tiles: keep it in L2 ahead of the streaming A rows and C
      // output.  CTA pairs (banded walk): keep A with this policy, B at normal priority.
      const uint64_t pol_b = l2_policy_evict_last();
      const uint64_t pol_n = l2_policy_evict_normal();
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      bool ok = true;
      TileCoord tc;
      for (int64_t t = tile0; ok && t < total_tiles; t += tile_stride) {
        if (!sched.locate(args, t, tc)) break;
        const int32_t a_row = (int32_t)(tc.m0 + C::ROWS * rank);
        const int32_t b_row = tc.be * args.N + tc.n0 + C::B_ROWS * rank;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_sleep(empty_bar(stage), phase ^ 1, abort)) {
            record_error(args.err, DEV_TIMEOUT, abort);
            ok = false;
            break;
          }
          if constexpr (C::CG == 1) {
            mbar_arrive_expect_tx(full_bar(stage), C::STAGE_TX);
            tma_load_2d(sA + stage * C::A_STAGE, &tmA, kb * BK, a_row, full_bar(stage));
            tma_load_2d_hint(sB + stage * C::B_STAGE, &tmB, kb * BK, b_row, full_bar(stage),
                             pol_b);
          } else {
            // both CTAs' bytes are counted on the leader's barrier
            const uint32_t bar = mapa_shared(full_bar(stage), 0);
            if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), C::STAGE_TX);
            // (banded walk: A is the operand the tiles in flight reuse, B streams)
            tma_load_2d_pair_hint(sA + stage * C::A_STAGE, &tmA, kb * BK, a_row, bar, pol_b);
            tma_load_2d_pair_hint(sB + stage * C::B_STAGE, &tmB, kb * BK, b_row, bar, pol_n);
            if constexpr (C::ASYM) {
              // the peer's A rows (after the leader's ROWS) and its half of B, into the peer's
              // shared memory at the same offsets, counted on this barrier
              tma_load_2d_mc_pair_hint(sA + stage * C::A_STAGE, &tmA, kb * BK, a_row + C::ROWS,
                                       full_bar(stage), 0x2, pol_b);
              tma_load_2d_mc_pair_hint(sB + stage * C::B_STAGE, &tmB, kb * BK, b_row + C::B_ROWS,
                                       full_bar(stage), 0x2, pol_n);
            }
          }
          ++issued;
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
      }
      // Let this CTA's last loads land before it can exit.  In the leader they complete
      // its full barrier; in the peer, the MMA consuming them frees its empty barrier.
      const int64_t pending = issued < C::STAGES ? issued : C::STAGES;
      for (int64_t i = 0; i < pending; ++i) {
        stage = (stage + C::STAGES - 1) % C::STAGES;
        if (stage == C::STAGES - 1) phase ^= 1;
        if (rank == 0) mbar_wait_timed(full_bar(stage), phase);
        else mbar_wait_timed(empty_bar(stage), phase);
      }
    } else if (!C::ROLE4 && warp == C::MMA_WARP && lane == 0 && rank == 0) {
      // ================================ MMA issuer ================================
      // One thread, and the pace of the whole pipeline: per K block two barrier tests,
      // four MMAs and one commit, with the descriptors of every stage precomputed.
      GroupedScheduler<C::BM, C::BN, C::TILE_BAND> sched;
      const uint64_t adesc0 = kmajor_sw128_desc(sA);
      const uint64_t bdesc0 = kmajor_sw128_desc(sB);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      TileCoord tc;
      for (int64_t t = tile0; ok && t < total_tiles; t += tile_stride) {
        if (!sched.locate(args, t, tc)) break;
        for (int kb = 0; kb < KB; ++kb) {
          // operands first: they are usually in place well before the TMEM stage is free
          if (!mbar_wait_cg<C::CG>(full_bar(stage), phase, abort) ||
              !mbar_wait_cg<C::CG>(tempty_bar(acc), acc_phase ^ 1, abort)) {
            record_error(args.err, DEV_TIMEOUT, abort);
            ok = false;
            break;
          }
          tc_fence_after();
          issue_kblock<C>(tmem_base + acc * C::BN, adesc0 + ((stage * C::A_STAGE) >> 4),
                          bdesc0 + ((stage * C::B_STAGE) >> 4), empty_bar(stage));
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
          if (++acc == C::ACC_STAGES) { acc = 0; acc_phase ^= 1; }
        }
      }
      // Every MMA this thread issued has finished before TMEM is released.  A wait that
      // gives up is reported and waited out once more (bounded) before the teardown.
      if constexpr (C::CG == 1) umma_commit(smem_u32(&ctl->mma_done));
      else umma_commit_pair(smem_u32(&ctl->mma_done), 0x1);
      if (!mbar_wait_timed(smem_u32(&ctl->mma_done), 0)) {
        record_error(args.err, DEV_TIMEOUT, abort);
        mbar_wait_timed(smem_u32(&ctl->mma_done), 0);
      }
    }
    __syncwarp();
  } else {
    // ================================= epilogue =================================
    if constexpr (!C::SPARE_QUARTER) asm volatile("setmaxnreg.inc.sync.aligned.u32 232;");
    const uint32_t quarter = warp & 3;              // TMEM lanes 32*quarter .. +31
    const uint32_t half = C::column_half(warp);     // columns half*COLS .. +COLS-1
    const int nblk = args.N / 128;
    const float* a_scales = static_cast<const float*>(args.a_scales);
    const float* b_scales = static_cast<const float*>(args.b_scales);
    __nv_bfloat16* Cmat = static_cast<__nv_bfloat16*>(args.C);
    // the MMA CTA's barrier that collects "TMEM stage drained" from both CTAs
    auto tempty_mma = [&](int s) {
      return (C::CG == 2) ? mapa_shared(tempty_bar(s), 0) : tempty_bar(s);
    };
    GroupedScheduler<C::BM, C::BN, C::TILE_BAND> sched;
    // C rows go out as one 32-byte sector per lane when C allows it
    const bool c_vec32 = (reinterpret_cast<uintptr_t>(args.C) & 31) == 0;
    uint32_t acc_stage = 0, acc_phase = 0;  // TMEM partial ring
    uint32_t op_stage = 0, op_phase = 0;    // operand ring (its empty barriers)
    uint32_t rel = 0;                       // K blocks released so far (ROLE4: barrier rel % 4)
    // This warp has finished reading TMEM stage acc_stage: tell the MMA thread (in the MMA
    // CTA of a pair).
    auto release_stage = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0)
        mbar_arrive_cluster_or_local<C::CG>(tempty_mma(C::ROLE4 ? (int)(rel & 3) : (int)acc_stage));
    };
    bool ok = true;
    TileCoord tc;
    for (int64_t t = tile0; ok && t < total_tiles; t += tile_stride) {
      if (!sched.locate(args, t, tc)) break;
      const int64_t row = tc.m0 + C::ROWS * rank + quarter * 32 + lane;
      const bool row_in = row < args.M_total;
      const int col0 = tc.n0 + (int)half * C::COLS;  // first column of this warp
      // this warp's columns touch scale blocks col0/128 and (col0+COLS-1)/128 (<= 2)
      const int blk_lo = col0 / 128;
      const int blk_hi = (col0 + C::COLS - 1) / 128;
      const bool lo_in = blk_lo < nblk, hi_in = !C::ONE_BLOCK && blk_hi < nblk;
      // the group's expert, re-read per tile (kept out of the scheduler's live registers)
      const int64_t be = args.expert_ids ? ldg_s32(args.expert_ids + tc.e) : tc.e;
      // Scales: loaded two K blocks ahead of their use, a_scales[kb, row] (one load per lane,
      // consecutive K blocks M_total apart, their lines prefetched into L1 SCALE_LOOKAHEAD K
      // blocks ahead) and b_scales[be, blk, kb] (uniform per warp).  Every lane loads from a
      // valid address without a predicate: rows past M_total read row 0 and scale blocks past
      // N read block 0 (those results are never stored), and K blocks past the last re-read it.
      const float* sa_ptr = a_scales + (row_in ? row : 0);
      const float* sb_lo = b_scales + (be * nblk + (lo_in ? blk_lo : 0)) * KB;
      const float* sb_hi = b_scales + (be * nblk + (hi_in ? blk_hi : 0)) * KB;
      float2 acc[C::COLS / 2];  // columns 2j, 2j+1
#pragma unroll
      for (int j = 0; j < C::COLS / 2; ++j) acc[j] = make_float2(0.0f, 0.0f);
      for (int k = 2; k < C::SCALE_LOOKAHEAD && k < KB; ++k)
        prefetch_l1(sa_ptr + (int64_t)k * args.M_total);
      // K block kb's values (sa_n, sbl_n, sbh_n) and K block kb + 1's (sa_2, ...)
      const int kb1 = KB > 1 ? 1 : 0;
      float sa_n = ldg_f32(sa_ptr);
      float sbl_n = ldg_f32(sb_lo);
      float sbh_n = C::ONE_BLOCK ? 0.0f : ldg_f32(sb_hi);
      float sa_2 = ldg_f32(sa_ptr + (int64_t)kb1 * args.M_total);
      float sbl_2 = ldg_f32(sb_lo + kb1);
      float sbh_2 = C::ONE_BLOCK ? 0.0f : ldg_f32(sb_hi + kb1);
      const uint32_t taddr0 = tmem_base + ((quarter * 32) << 16) + half * C::COLS;
      // unrolled by two: the next K block's scale products and loads schedule into the tail
      // of this one's promotion (~1 % faster on the skewed 64-expert and dense 8192^3 GEMMs)
#pragma unroll 2
      for (int kb = 0; kb < KB; ++kb) {
        const float s_lo = sa_n * sbl_n;
        const float s_hi = C::ONE_BLOCK ? s_lo : sa_n * sbh_n;
        sa_n = sa_2;
        sbl_n = sbl_2;
        sbh_n = sbh_2;
        const int kp = kb + C::SCALE_LOOKAHEAD < KB ? kb + C::SCALE_LOOKAHEAD : KB - 1;
        prefetch_l1(sa_ptr + (int64_t)kp * args.M_total);
        const int k2 = kb + 2 < KB ? kb + 2 : KB - 1;
        sa_2 = ldg_f32(sa_ptr + (int64_t)k2 * args.M_total);
        sbl_2 = ldg_f32(sb_lo + k2);
        if constexpr (!C::ONE_BLOCK) sbh_2 = ldg_f32(sb_hi + k2);
        // the K block's MMAs are done when its operand stage's empty barrier completes
        const bool got = __all_sync(
            0xffffffffu, mbar_wait_cg<C::CG>(empty_bar(op_stage), op_phase, abort));
        if (!got) {
          if (lane == 0) record_error(args.err, DEV_TIMEOUT, abort);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = taddr0 + acc_stage * C::BN;
        // 16-column chunks never straddle a 128-column scale block
        auto chunk_scale = [&](int c) { return ((col0 + 16 * c) / 128 == blk_lo) ? s_lo : s_hi; };
        if constexpr (C::LOAD_ALL) {
          uint32_t p[C::CHUNKS][16];
#pragma unroll
          for (int c = 0; c < C::CHUNKS; ++c) tmem_ld_32x32b_x16(taddr + 16 * c, p[c]);
          tmem_ld_wait();
          release_stage();
#pragma unroll
          for (int c = 0; c < C::CHUNKS; ++c) promote16(acc + 8 * c, p[c], chunk_scale(c));
        } else {
          // 64-column halves: load, promote, ..., load the last half, release, promote
          uint32_t p[64];
#pragma unroll
          for (int h = 0; h < C::COLS / 64; ++h) {
            tmem_ld_32x32b_x64(taddr + 64 * h, p);
            tmem_ld_wait();
            if (h == C::COLS / 64 - 1) release_stage();
            promote16(acc + 32 * h + 0, p, chunk_scale(4 * h + 0));
            promote16(acc + 32 * h + 8, p + 16, chunk_scale(4 * h + 1));
            promote16(acc + 32 * h + 16, p + 32, chunk_scale(4 * h + 2));
            promote16(acc + 32 * h + 24, p + 48, chunk_scale(4 * h + 3));
          }
        }
        if (++acc_stage == C::ACC_STAGES) { acc_stage = 0; acc_phase ^= 1; }
        if (++op_stage == C::STAGES) { op_stage = 0; op_phase ^= 1; }
        ++rel;
      }
      if (!ok) break;
      if (row < tc.m_end) {
        // C is written once and not read again here: first out of L2
        const uint64_t pol_c = l2_policy_evict_first();
        __nv_bfloat16* dst = Cmat + row * (int64_t)args.N + col0;
#pragma unroll
        for (int c = 0; c < C::CHUNKS; ++c) {
          if (col0 + 16 * c < args.N) {  // the last column tile may pass N
            const float2* a = acc + 8 * c;
            uint32_t v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = pack_bf16x2(a[j].x, a[j].y);
            // N % 128 == 0 and col0 % 16 == 0: dst + 16c is 32-byte aligned when C is
            if (c_vec32) {
              st_global_v8_hint(dst + 16 * c, v, pol_c);
            } else {
              st_global_v4_hint(dst + 16 * c, v[0], v[1], v[2], v[3], pol_c);
              st_global_v4_hint(dst + 16 * c + 8, v[4], v[5], v[6], v[7], pol_c);
            }
          }
        }
      }
    }
  }

  // ---- teardown ------------------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  // the pair's MMAs and remote arrivals are finished before either CTA frees TMEM or exits
  if constexpr (C::CG == 2) cluster_sync();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc<C::CG>(tmem_base, TMEM_COLS);
  }
}

template <class C>
cudaError_t launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& args,
                   int num_sms, cudaStream_t stream) {
  static_assert(smem_bytes<C>() <= 227 * 1024, "shared memory per CTA");
  static std::atomic<bool> attr_set[64];  // per device; several host threads may launch
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(bsfp8_blockwise_kernel<C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes<C>());
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set[dev].store(true, std::memory_order_release);
  }
  // Upper bound of the tile count known on the host (offsets live on the device).
  const int64_t max_row_tiles = (args.M_total + C::BM - 1) / C::BM + args.E;
  const int64_t max_tiles = max_row_tiles * ((args.N + C::BN - 1) / C::BN);
  const int64_t pairs = num_sms / C::CG;
  const int grid = (int)((max_tiles < pairs ? max_tiles : pairs) * C::CG);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = smem_bytes<C>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C::CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bsfp8_blockwise_kernel<C>, tmA, tmB, args);
}

// 1-CTA 128 x 256 (2 TMEM stages), CTA pair 256 x 256 (2 stages), CTA pair 256 x 160
// (3 stages), CTA pair 256 x 128 (4 stages), 1-CTA 128 x 128 (4 stages).  With 160 or 128
// columns each epilogue warp loads all of its columns at once and frees the stage early.
// 1-CTA 96 x 256 and CTA pair 192 x 256: 96 A rows per CTA, role warps on their own SMSP.
using Cta1x256 = Cfg<1, 256, 4, 2>;
using Pair256 = Cfg<2, 256, 6, 2>;
using Pair160 = Cfg<2, 160, 8, 3>;
using Pair128 = Cfg<2, 128, 8, 4>;
using Cta1x128 = Cfg<1, 128, 4, 4>;
using Cta1x96x256 = Cfg<1, 256, 5, 2, 96>;
using Pair192x256 = Cfg<2, 256, 6, 2, 96>;
using Cta1x96x192 = Cfg<1, 192, 5, 2, 96>;
using Pair192x192 = Cfg<2, 192, 7, 2, 96>;
using Cta1x128x192 = Cfg<1, 192, 4, 2, 128>;
using Pair224x256 = Cfg<2, 256, 6, 2, 96, 128>;

}  // namespace bw

int blockwise_b_rows(BlockwiseTile tile) {
  switch (tile) {
    case TILE_CTA1_256: return bw::Cta1x256::B_ROWS;
    case TILE_PAIR_256: return bw::Pair256::B_ROWS;
    case TILE_PAIR_160: return bw::Pair160::B_ROWS;
    case TILE_PAIR_128: return bw::Pair128::B_ROWS;
    case TILE_CTA1_128: return bw::Cta1x128::B_ROWS;
    case TILE_CTA1_96: return bw::Cta1x96x256::B_ROWS;
    case TILE_PAIR_192: return bw::Pair192x256::B_ROWS;
    case TILE_CTA1_96x192: return bw::Cta1x96x192::B_ROWS;
    case TILE_PAIR_192x192: return bw::Pair192x192::B_ROWS;
    case TILE_CTA1_128x192: return bw::Cta1x128x192::B_ROWS;
    case TILE_PAIR_224: return bw::Pair224x256::B_ROWS;
  }
  return 0;
}

int blockwise_a_rows(BlockwiseTile tile) {
  switch (tile) {
    case TILE_CTA1_96: return bw::Cta1x96x256::ROWS;
    case TILE_PAIR_192: return bw::Pair192x256::ROWS;
    case TILE_CTA1_96x192: return bw::Cta1x96x192::ROWS;
    case TILE_PAIR_192x192: return bw::Pair192x192::ROWS;
    case TILE_PAIR_224: return bw::Pair224x256::A_BOX;
    default: return 128;
  }
}

cudaError_t launch_bsfp8_blockwise(BlockwiseTile tile, const CUtensorMap& tmA,
                                   const CUtensorMap& tmB, const GemmArgs& args, int num_sms,
                                   cudaStream_t stream) {
  switch (tile) {
    case TILE_CTA1_256: return bw::launch<bw::Cta1x256>(tmA, tmB, args, num_sms, stream);
    case TILE_PAIR_256: return bw::launch<bw::Pair256>(tmA, tmB, args, num_sms, stream);
    case TILE_PAIR_160: return bw::launch<bw::Pair160>(tmA, tmB, args, num_sms, stream);
    case TILE_PAIR_128: return bw::launch<bw::Pair128>(tmA, tmB, args, num_sms, stream);
    case TILE_CTA1_128: return bw::launch<bw::Cta1x128>(tmA, tmB, args, num_sms, stream);
    case TILE_CTA1_96: return bw::launch<bw::Cta1x96x256>(tmA, tmB, args, num_sms, stream);
    case TILE_PAIR_192: return bw::launch<bw::Pair192x256>(tmA, tmB, args, num_sms, stream);
    case TILE_CTA1_96x192: return bw::launch<bw::Cta1x96x192>(tmA, tmB, args, num_sms, stream);
    case TILE_PAIR_192x192: return bw::launch<bw::Pair192x192>(tmA, tmB, args, num_sms, stream);
    case TILE_CTA1_128x192: return bw::launch<bw::Cta1x128x192>(tmA, tmB, args, num_sms, stream);
    case TILE_PAIR_224: return bw::launch<bw::Pair224x256>(tmA, tmB, args, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bsfp8

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
// Roles (12 warps per CTA): warp 0 TMA producer (own 128 token rows, own 128 weight rows);
// warp 1 TMEM owner and, in CTA 0 of the pair, the MMA thread (per 128-K block tcgen05.cp
// of its scale blocks and 4 x tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale; one
// commit per ring stage, multicast to both CTAs); warp 2 scale loader; warps 4-11 epilogue
// (TMEM lane quarter w%4, column half (w-4)/4, 32-column subtiles).
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

constexpr int BK = 128;
constexpr int BM = 256;        // token rows per pair tile (128 per CTA)
constexpr int BN = 256;        // weight rows per pair tile (MMA N)
constexpr int EPI_N = 32;      // epilogue subtile columns
// Tiles are walked in bands of 16 row tiles (row index fastest inside a band): the 76 pairs
// in flight share ~5 columns of B, and B is read from DRAM about once per band
constexpr int TILE_BAND = 16;
constexpr int NUM_THREADS = 384;
constexpr int EPI_WARP0 = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr int SF_BLOCK = 512;  // packed scale block: 128 rows x 4 codes
// K blocks of 128 per ring stage (k_group_size of the per-K-stage context, MAX
// EpilogueWarpContext page, per_k_stage): one full/empty round trip and one commit per KG
// K blocks instead of per K block
constexpr int KG = 2;
constexpr int STAGES = 3;  // ring stages of KG K blocks (64 KB of operands each)
// Row-major scale copies in flight before the oldest is announced.  A stage's copies start
// once the MMA has freed it; announcing stage s only after the copies of s + L are issued
// waits for the MMA to free s + L, so L <= STAGES - 2 keeps that off the MMA's path.
constexpr int SCALE_LOOKAHEAD = 1;
static_assert(SCALE_LOOKAHEAD <= STAGES - 2, "scale announce would wait on the MMA");
constexpr TmemPlan PLAN = tmem_overlap_plan(BK, EPI_N, 32, true, BN, 512);
static_assert(PLAN.right_offset == 244 && PLAN.a_scale_offset == 500 &&
              PLAN.b_scale_offset == 504 && PLAN.early_release_subtile == 0,
              "plan for BLOCK_K 128, VEC 32");

constexpr uint32_t A_SUB = 128 * BK;   // one K block of this CTA's token rows
constexpr uint32_t B_SUB = 128 * BK;   // one K block of this CTA's weight rows
constexpr uint32_t A_STAGE = KG * A_SUB;
constexpr uint32_t B_STAGE = KG * B_SUB;
constexpr uint32_t SMEM_A = 0;
constexpr uint32_t SMEM_B = SMEM_A + STAGES * A_STAGE;
constexpr uint32_t SFA_STAGE = KG * SF_BLOCK;                        // 1 block per K block
constexpr uint32_t SFB_STAGE = KG * 2 * SF_BLOCK;                    // 2 blocks per K block
constexpr uint32_t SMEM_SFA = SMEM_B + STAGES * B_STAGE;
constexpr uint32_t SMEM_SFB = SMEM_SFA + STAGES * SFA_STAGE;
// Scale staging for the grouped loader: per group of 4 stages, 16 bytes (4 stages x 4
// codes) of each of this CTA's 128 token rows and the tile's 256 weight rows.
constexpr int GROUP = 4;
constexpr uint32_t STG_A = 128 * 16;
constexpr uint32_t STG_SLOT = STG_A + 256 * 16;
constexpr int STG_SLOTS = 3;
constexpr uint32_t SMEM_STG = SMEM_SFB + STAGES * SFB_STAGE;
constexpr uint32_t SMEM_CTL = SMEM_STG + STG_SLOTS * STG_SLOT;
constexpr uint32_t SUB_TX = 2 * (A_SUB + B_SUB);  // both CTAs' bytes of one K block
static_assert(GROUP % KG == 0, "a grouped scale fetch covers whole ring stages");

struct Ctl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
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
constexpr uint32_t SMEM_BYTES = SMEM_CTL + sizeof(Ctl) + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

__device__ __forceinline__ void record_error(int* err, int code, volatile int* abort) {
  atomicCAS(err, 0, code);
  *abort = 1;
}

__device__ __forceinline__ uint64_t sf_block_desc(uint32_t saddr) {
  return make_smem_desc(saddr, 0, 128, LAYOUT_NONE);
}

// PACKED_B: weight scales pre-packed in [E][N/128][K/128] blocks of 512 bytes (else
// row-major [E, N, K/32]); an instantiation each, so the row-major loader carries no branch.
template <bool PACKED_B>
__global__ void __launch_bounds__(NUM_THREADS, 1)
bsmxfp8_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + SMEM_CTL);
  volatile int* abort = &ctl->abort;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const int KB = args.K / BK;
  const int scale_row = args.K / 32;
  const uint32_t rank = cluster_ctarank();
  const int64_t tile0 = blockIdx.x / 2;
  const int64_t tile_stride = gridDim.x / 2;

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
      mbar_init(full_bar(s), 3);   // leader producer (+ both CTAs' bytes) + 2 scale loaders
      mbar_init(empty_bar(s), 1);  // one (multicast) MMA commit
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(accf_bar(s), 1);
      mbar_init(acce_bar(s), NUM_EPI_WARPS * 2);
    }
    mbar_init(ovl_bar, NUM_EPI_WARPS);  // the 4 overlap-owning warps of each CTA
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
            // this K block's scales into the TMEM scale columns (after the previous K block's
            // MMAs, which read them, in this thread's issue order)
            const uint32_t sfa_s = sSFA + stage * SFA_STAGE + u * SF_BLOCK;
            const uint32_t sfb_s = sSFB + stage * SFB_STAGE + u * 2 * SF_BLOCK;
            tmem_cp_32x128b_warpx4<2>(sfa_t, sf_block_desc(sfa_s));
            tmem_cp_32x128b_warpx4<2>(sfb_t, sf_block_desc(sfb_s));
            tmem_cp_32x128b_warpx4<2>(sfb_t + 4, sf_block_desc(sfb_s + SF_BLOCK));
            const uint64_t adesc = kmajor_sw128_desc(sA + stage * A_STAGE + u * A_SUB);
            const uint64_t bdesc = kmajor_sw128_desc(sB + stage * B_STAGE + u * B_SUB);
#pragma unroll
            for (int k = 0; k < BK / 32; ++k)
              umma_mxf8f6f4<2>(d_tmem, adesc + (uint64_t)(k * 2), bdesc + (uint64_t)(k * 2),
                               idesc_mxf8f6f4_e4m3(BM, BN, k, k), sfa_t, sfb_t,
                               (kb0 + u > 0 || k > 0) ? 1u : 0u);
          }
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
  } else if (warp == 2) {
    // =============================== scale loader ===============================
    // Per stage: this CTA's 128 token rows (one packed block) and all 256 weight rows of
    // the tile (two packed blocks, duplicated in both CTAs: the pair MMA reads the weight
    // scales from each CTA's own TMEM).  Announced on the MMA CTA's full barrier.
    const uint8_t* a_sc = static_cast<const uint8_t*>(args.a_scales);
    const uint8_t* b_sc = static_cast<const uint8_t*>(args.b_scales);
    // weight scales either row-major [E, N, K/32] or pre-packed [E][N/128][K/128] blocks
    constexpr bool packed_b = PACKED_B;
    const int nblk = args.N / 128;
    GroupedScheduler<BM, BN, TILE_BAND> sched;
    uint32_t stage = 0, phase = 0;
    // Grouped path: when a row's codes for 4 consecutive stages form one aligned 16-byte
    // chunk (K % 512 == 0, 16-byte aligned scale arrays), fetch a 4-stage group per row with
    // one 16-byte copy, two groups ahead, and transpose each stage's words into its packed
    // blocks in shared memory.
    const bool grouped = (args.K % (GROUP * BK) == 0) &&
                         (reinterpret_cast<uintptr_t>(a_sc) % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(b_sc) % 16 == 0);
    if (grouped) {
      const int G = KB / GROUP;  // groups per tile
      const uint32_t sSTG = smem_u32(smem + SMEM_STG);
      const uint8_t* stg = smem + SMEM_STG;
      GroupedScheduler<BM, BN, TILE_BAND> pre;
      TileCoord tp;
      int64_t tp_t = tile0;
      bool pre_ok = pre.locate(args, tp_t, tp);
      int qp = 0;
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
              const int r = 32 * i + (int)lane;
              const int n = tp.n0 + r;
              const bool live = n < args.N;
              const uint8_t* src = b_sc + ((int64_t)tp.be * args.N + n) * scale_row + 16 * qp;
              cp_async_16(dst + STG_A + r * 16, live ? src : b_sc, live ? 16u : 0u);
            }
          }
          if (++qp == G) {
            qp = 0;
            tp_t += tile_stride;
            pre_ok = tp_t < total_tiles && pre.locate(args, tp_t, tp);
          }
        }
        cp_async_commit();  // an empty group keeps the group count in step
      };
      issue_group(0);
      issue_group(1);
      int64_t g = 0;
      bool ok = true;
      TileCoord tc;
      for (int64_t t = tile0; ok && t < total_tiles; t += tile_stride) {
        if (!sched.locate(args, t, tc)) break;
        for (int q = 0; ok && q < G; ++q, ++g) {
          cp_async_wait_group<1>();  // group g has landed (g + 1 may be in flight)
          __syncwarp();
          const uint8_t* src = stg + (g % STG_SLOTS) * STG_SLOT;
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
            // packed block: row r = 32*rg + lane at byte lane*16 + rg*4
            auto gather = [&](const uint8_t* rows) {
              uint4 w;
              w.x = *reinterpret_cast<const uint32_t*>(rows + (0 * 32 + lane) * 16 + 4 * j);
              w.y = *reinterpret_cast<const uint32_t*>(rows + (1 * 32 + lane) * 16 + 4 * j);
              w.z = *reinterpret_cast<const uint32_t*>(rows + (2 * 32 + lane) * 16 + 4 * j);
              w.w = *reinterpret_cast<const uint32_t*>(rows + (3 * 32 + lane) * 16 + 4 * j);
              return w;
            };
            *reinterpret_cast<uint4*>(smem + SMEM_SFA + stage * SFA_STAGE + u * SF_BLOCK +
                                      lane * 16) = gather(src);
            uint4* sfb =
                reinterpret_cast<uint4*>(smem + SMEM_SFB + stage * SFB_STAGE + u * 2 * SF_BLOCK);
            if constexpr (packed_b) {
              const uint8_t* pb = src + STG_A + j * SF_BLOCK + lane * 16;
              sfb[lane] = *reinterpret_cast<const uint4*>(pb);
              sfb[32 + lane] = *reinterpret_cast<const uint4*>(pb + 4 * SF_BLOCK);
            } else {
              sfb[lane] = gather(src + STG_A);
              sfb[32 + lane] = gather(src + STG_A + 128 * 16);
            }
            }
            fence_proxy_async_smem();  // generic-proxy writes -> tcgen05.cp (async proxy)
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(full_bar(stage), 0));
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          __syncwarp();
          issue_group((int)((g + 2) % STG_SLOTS));  // the slot group g - 1 used is free
        }
      }
      cp_async_wait_group<0>();
    } else {
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
  } else if (warp >= EPI_WARP0) {
    // ================================= epilogue =================================
    const uint32_t ew = warp - EPI_WARP0;
    const uint32_t quarter = warp & 3;
    const uint32_t half = ew >> 2;  // accumulator columns half*128 .. +127
    __nv_bfloat16* Cmat = static_cast<__nv_bfloat16*>(args.C);
    GroupedScheduler<BM, BN, TILE_BAND> sched;
    const uint64_t pol_c = l2_policy_evict_first();
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
      for (int s = 0; s < 4; ++s) {
        const int sub = high_first ? 3 - s : s;
        const int col = (int)half * 128 + sub * EPI_N;  // column inside the tile
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + ((quarter * 32) << 16) + col_base + col, v);
        tmem_ld_wait();
        if (s == PLAN.early_release_subtile && owns_overlap) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(ovl_bar, 0));
        }
        const int n = tc.n0 + col;
        if (row < tc.m_end && n < args.N) {
          __nv_bfloat16* dst = Cmat + row * (int64_t)args.N + n;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            auto f = [&](int j) { return __uint_as_float(v[8 * q + j]); };
            st_global_v4_hint(dst + 8 * q, pack_bf16x2(f(0), f(1)), pack_bf16x2(f(2), f(3)),
                              pack_bf16x2(f(4), f(5)), pack_bf16x2(f(6), f(7)), pol_c);
          }
        }
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
template <bool PACKED_B>
cudaError_t launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& args,
                   int num_sms, cudaStream_t stream) {
  static std::atomic<bool> attr_set[64];  // per device; several host threads may launch
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(bsmxfp8_pair_kernel<PACKED_B>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set[dev].store(true, std::memory_order_release);
  }
  const int64_t max_row_tiles = (args.M_total + mxp::BM - 1) / mxp::BM + args.E;
  const int64_t max_tiles = max_row_tiles * ((args.N + mxp::BN - 1) / mxp::BN);
  const int64_t pairs = num_sms / 2;
  const int grid = (int)((max_tiles < pairs ? max_tiles : pairs) * 2);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(mxp::NUM_THREADS);
  cfg.dynamicSmemBytes = mxp::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bsmxfp8_pair_kernel<PACKED_B>, tmA, tmB, args);
}
}  // namespace mxp

cudaError_t launch_bsmxfp8_pair(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                const GemmArgs& args, int num_sms, cudaStream_t stream) {
  return args.b_scales_packed ? mxp::launch<true>(tmA, tmB, args, num_sms, stream)
                              : mxp::launch<false>(tmA, tmB, args, num_sms, stream);
}

TmemPlan mx_pair_tmem_plan() { return mxp::PLAN; }

}  // namespace bsfp8

// Blockwise-scaled FP8 grouped GEMM for sm_103a (one CTA per SM, persistent).
//
//   C[m, n] = sum_kb a_scales[kb, m] * b_scales[e, n/128, kb] * sum_{k in kb} A[m,k] B[e,n,k]
//
// with e the expert owning row m, 1x128 A scales and 128x128 B scales over K blocks of
// 128, fp32 accumulation and bf16 output.
//
// Structure (prior art: promote_accumulators in MAX kernels grouped_matmul_sm100_blockwise_fp8
// -- per-K-block TMEM partials promoted with a_scale x b_scale into fp32 register tiles;
// EpilogueWarpContext in MAX sm100_structured -- epilogue warps consuming a TMEM stage ring
// per K stage; the warp-specialized partitions of the Triton Gluon example "Overlapping
// Accumulator Block-Scaled Matrix Multiplication"):
//
//   warp 0       TMA producer: per K block, A tile [128 x 128] and B tile [256 x 128]
//                (e4m3, 128-byte swizzle) into a 4-stage shared-memory ring.
//   warp 1       TMEM owner + MMA issuer: per K block, 4 x tcgen05.mma kind::f8f6f4
//                (M=128, N=256, K=32) into a fresh TMEM partial (2-stage ring, 2 x 256
//                columns = all 512); commits release the SMEM stage and publish the partial.
//   warps 4-11   epilogue: warp w reads TMEM lanes 32*(w%4).. (its rows) and columns
//                128*((w-4)/4).. (its column half); per K block it loads the fp32 partial,
//                releases the TMEM stage and promotes acc = fma(sa*sb, partial, acc) in
//                registers (128 per thread); after the last K block it rounds to bf16 and
//                stores the rows that belong to the tile's expert.
//
// The A and B scales are read by the epilogue from global memory one K block ahead (the
// page reads b_scale from global memory and stages the A-scale strip in SMEM; here both
// come through the read-only cache, which keeps the SMEM ring free for operands).
#include <cuda_bf16.h>
#include "common.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace bsfp8 {
namespace bw {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;
constexpr int STAGES = 4;
constexpr int ACC_STAGES = 2;
constexpr int NUM_THREADS = 384;
constexpr int EPI_WARP0 = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr int COLS_PER_WARP = BN / 2;  // two epilogue warps share each 32-lane quarter
constexpr uint32_t TMEM_COLS = 512;
static_assert(ACC_STAGES * BN <= (int)TMEM_COLS, "TMEM ring too large");

constexpr uint32_t A_STAGE = BM * BK;  // 16 KB
constexpr uint32_t B_STAGE = BN * BK;  // 32 KB
constexpr uint32_t SMEM_A = 0;
constexpr uint32_t SMEM_B = SMEM_A + STAGES * A_STAGE;
constexpr uint32_t SMEM_CTL = SMEM_B + STAGES * B_STAGE;

struct Ctl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[ACC_STAGES];
  uint64_t tempty[ACC_STAGES];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  int valid;
  int pad;
  long long total_tiles;
};
constexpr uint32_t SMEM_BYTES = SMEM_CTL + sizeof(Ctl) + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

constexpr uint32_t IDESC = idesc_f8f6f4_e4m3(BM, BN);

__device__ __forceinline__ void record_error(int* err, int code, volatile int* abort) {
  atomicCAS(err, 0, code);
  *abort = 1;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
bsfp8_blockwise_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB, const GemmArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + SMEM_CTL);
  volatile int* abort = &ctl->abort;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const int KB = args.K / BK;

  // ---- work discovery: validate the offsets, count tiles -------------------------------
  if (warp == 0) {
    int ok;
    int64_t row_tiles;
    validate_offsets<BM>(args.offsets, args.E, args.M_total, ok, row_tiles);
    if (lane == 0) {
      ctl->valid = ok;
      ctl->total_tiles = row_tiles * ((args.N + BN - 1) / BN);
      ctl->abort = 0;
      if (!ok && blockIdx.x == 0) atomicCAS(args.err, 0, DEV_BAD_OFFSETS);
    }
  }
  __syncthreads();
  const int64_t total_tiles = ctl->total_tiles;
  if (!ctl->valid || (int64_t)blockIdx.x >= total_tiles) return;

  // ---- setup: barriers, TMEM ---------------------------------------------------------
  const uint32_t sA = smem_u32(smem + SMEM_A);
  const uint32_t sB = smem_u32(smem + SMEM_B);
  auto full_bar = [&](int s) { return smem_u32(&ctl->full[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&ctl->empty[s]); };
  auto tfull_bar = [&](int s) { return smem_u32(&ctl->tfull[s]); };
  auto tempty_bar = [&](int s) { return smem_u32(&ctl->tempty[s]); };

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int s = 0; s < ACC_STAGES; ++s) {
      mbar_init(tfull_bar(s), 1);
      mbar_init(tempty_bar(s), NUM_EPI_WARPS);
    }
    mbar_init(smem_u32(&ctl->mma_done), 1);
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc<1>(smem_u32(&ctl->tmem_base), TMEM_COLS);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp < EPI_WARP0) {
    // warpgroup 0: producer, MMA issuer and two idle warps give registers away
    asm volatile("setmaxnreg.dec.sync.aligned.u32 40;");
    if (warp == 0) {
    // =============================== TMA producer ===============================
    if (lane == 0) {
      GroupedScheduler<BM, BN> sched(args.offsets, args.E, args.N);
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      bool ok = true;
      TileCoord tc;
      for (int64_t t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
        if (!sched.locate(t, tc)) break;
        const int32_t a_row = (int32_t)tc.m0;
        const int32_t b_row = tc.e * args.N + tc.n0;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1, abort)) {
            record_error(args.err, DEV_TIMEOUT, abort);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), A_STAGE + B_STAGE);
          tma_load_2d(sA + stage * A_STAGE, &tmA, kb * BK, a_row, full_bar(stage));
          tma_load_2d(sB + stage * B_STAGE, &tmB, kb * BK, b_row, full_bar(stage));
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      // Let the last loads land before the CTA can exit (they are complete already on
      // the normal path; after an abort they finish within microseconds).
      const int64_t pending = issued < STAGES ? issued : STAGES;
      for (int64_t i = 0; i < pending; ++i) {
        stage = (stage + STAGES - 1) % STAGES;
        if (stage == STAGES - 1) phase ^= 1;
        mbar_wait_timed(full_bar(stage), phase);
      }
    }
    __syncwarp();
    } else if (warp == 1) {
    // ================================ MMA issuer ================================
    if (lane == 0) {
      GroupedScheduler<BM, BN> sched(args.offsets, args.E, args.N);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      TileCoord tc;
      for (int64_t t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
        if (!sched.locate(t, tc)) break;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1, abort) ||
              !mbar_wait(full_bar(stage), phase, abort)) {
            record_error(args.err, DEV_TIMEOUT, abort);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * BN;
          const uint64_t adesc = kmajor_sw128_desc(sA + stage * A_STAGE);
          const uint64_t bdesc = kmajor_sw128_desc(sB + stage * B_STAGE);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)  // K = 32 e4m3 per instruction, 32 bytes
            umma_f8f6f4<1>(d_tmem, adesc + (uint64_t)(k * 2), bdesc + (uint64_t)(k * 2), IDESC,
                           k > 0 ? 1u : 0u);
          umma_commit(empty_bar(stage));  // operands consumed -> stage free
          umma_commit(tfull_bar(acc));    // partial ready for the epilogue
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
          if (++acc == ACC_STAGES) { acc = 0; acc_phase ^= 1; }
        }
      }
      // Every MMA this thread issued has finished before TMEM is released.
      umma_commit(smem_u32(&ctl->mma_done));
      mbar_wait_timed(smem_u32(&ctl->mma_done), 0);
    }
    __syncwarp();
    }
  } else {
    // ================================= epilogue =================================
    asm volatile("setmaxnreg.inc.sync.aligned.u32 232;");
    const uint32_t ew = warp - EPI_WARP0;
    const uint32_t quarter = warp & 3;         // TMEM lanes 32*quarter .. +31
    const uint32_t half = ew >> 2;             // columns half*128 .. +127
    const int nblk = args.N / 128;
    const float* a_scales = static_cast<const float*>(args.a_scales);
    const float* b_scales = static_cast<const float*>(args.b_scales);
    __nv_bfloat16* C = static_cast<__nv_bfloat16*>(args.C);
    GroupedScheduler<BM, BN> sched(args.offsets, args.E, args.N);
    uint32_t acc_stage = 0, acc_phase = 0;
    bool ok = true;
    TileCoord tc;
    for (int64_t t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
      if (!sched.locate(t, tc)) break;
      const int64_t row = tc.m0 + quarter * 32 + lane;
      const bool row_in = row < args.M_total;
      // N % 256 == 128: the second half of the last column tile is past N
      const bool cols_in = tc.n0 + (int)half * COLS_PER_WARP < args.N;
      const float* sa_ptr = a_scales + (row_in ? row : 0);
      const float* sb_ptr =
          cols_in ? b_scales + ((int64_t)tc.e * nblk + (tc.n0 + half * COLS_PER_WARP) / 128) * KB
                  : b_scales;
      float acc[COLS_PER_WARP];
#pragma unroll
      for (int j = 0; j < COLS_PER_WARP; ++j) acc[j] = 0.0f;
      float sa_next = row_in ? ldg_f32(sa_ptr) : 0.0f;
      float sb_next = ldg_f32(sb_ptr);
      for (int kb = 0; kb < KB; ++kb) {
        const float s = sa_next * sb_next;
        if (kb + 1 < KB) {
          sa_next = row_in ? ldg_f32(sa_ptr + (int64_t)(kb + 1) * args.M_total) : 0.0f;
          sb_next = cols_in ? ldg_f32(sb_ptr + kb + 1) : 0.0f;
        }
        const bool got = __all_sync(0xffffffffu, mbar_wait(tfull_bar(acc_stage), acc_phase, abort));
        if (!got) {
          if (lane == 0) record_error(args.err, DEV_TIMEOUT, abort);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr =
            tmem_base + ((quarter * 32) << 16) + acc_stage * BN + half * COLS_PER_WARP;
        uint32_t p0[32], p1[32];
        tmem_ld_32x32b_x32(taddr + 0, p0);
        tmem_ld_32x32b_x32(taddr + 32, p1);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          acc[j] = fmaf(s, __uint_as_float(p0[j]), acc[j]);
          acc[32 + j] = fmaf(s, __uint_as_float(p1[j]), acc[32 + j]);
        }
        tmem_ld_32x32b_x32(taddr + 64, p0);
        tmem_ld_32x32b_x32(taddr + 96, p1);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(acc_stage));
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          acc[64 + j] = fmaf(s, __uint_as_float(p0[j]), acc[64 + j]);
          acc[96 + j] = fmaf(s, __uint_as_float(p1[j]), acc[96 + j]);
        }
        if (++acc_stage == ACC_STAGES) { acc_stage = 0; acc_phase ^= 1; }
      }
      if (!ok) break;
      if (row < tc.m_end && cols_in) {
        __nv_bfloat16* dst = C + row * (int64_t)args.N + tc.n0 + half * COLS_PER_WARP;
#pragma unroll
        for (int j = 0; j < COLS_PER_WARP / 8; ++j)
          st_global_v4(dst + 8 * j, pack_bf16x2(acc[8 * j + 0], acc[8 * j + 1]),
                       pack_bf16x2(acc[8 * j + 2], acc[8 * j + 3]),
                       pack_bf16x2(acc[8 * j + 4], acc[8 * j + 5]),
                       pack_bf16x2(acc[8 * j + 6], acc[8 * j + 7]));
      }
    }
  }

  // ---- teardown ------------------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<1>(tmem_base, TMEM_COLS);
  }
}

}  // namespace bw

cudaError_t launch_bsfp8_blockwise(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                   const GemmArgs& args, int num_sms, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(bw::bsfp8_blockwise_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bw::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  // Upper bound of the tile count known on the host (offsets live on the device).
  const int64_t max_row_tiles = (args.M_total + bw::BM - 1) / bw::BM + args.E;
  const int64_t max_tiles = max_row_tiles * ((args.N + bw::BN - 1) / bw::BN);
  const int grid = (int)(max_tiles < num_sms ? max_tiles : num_sms);
  bw::bsfp8_blockwise_kernel<<<grid, bw::NUM_THREADS, bw::SMEM_BYTES, stream>>>(tmA, tmB, args);
  return cudaGetLastError();
}

}  // namespace bsfp8

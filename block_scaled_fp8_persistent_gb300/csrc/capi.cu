// C-ABI entry points: argument checks on the host, tensor-map encoding, kernel launch.
// Declarations and the contract live in include/bsfp8.h.
#include <algorithm>
#include <cstdlib>
#include <cmath>
#include <cstring>
#include <mutex>

#include "bsfp8.h"
#include "common.cuh"
#include "ptx.cuh"

namespace bsfp8 {

// One device error word per device (static device memory: nothing is allocated).
__device__ int g_error_word;

// Failure-detection check: one thread waits, with the GEMM kernels' bounded wait, for a
// phase of an mbarrier that nothing arrives on; when the wait gives up after limit_ns it
// records DEV_TIMEOUT in the device error word, as a GEMM kernel whose pipeline stalled
// would, and the kernel returns.
__global__ void wait_timeout_check_kernel(int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(smem_u32(&bar), 1);
  fence_mbarrier_init();
  if (!mbar_wait(smem_u32(&bar), 0, &abort_flag, limit_ns)) atomicCAS(err, 0, DEV_TIMEOUT);
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int num_sms = 0;
  int* err_word = nullptr;
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Device properties and the error word's address, once per device.
bsfp8_status device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BSFP8_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return BSFP8_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    d.num_sms = sms;
    if (d.supported) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return BSFP8_ERR_CUDA;
      d.err_word = static_cast<int*>(p);
    }
    d.ready = true;
  }
  if (!d.supported) return BSFP8_ERR_UNSUPPORTED_DEVICE;
  *out = &d;
  return BSFP8_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// 2D uint8 tensor map over a row-major [rows, inner] byte matrix, box [box_rows, box_inner],
// swizzled over box_inner bytes (128 or 64: the 128- or 64-byte swizzle), or with no swizzle
// (swizzle == false).
bool encode_u8_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                  uint32_t box_inner, uint32_t box_rows, bool swizzle = true) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            !swizzle ? CU_TENSOR_MAP_SWIZZLE_NONE
                     : box_inner == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D tensor map over packed e2m1 [rows, K] (K/2 bytes per row, 32-byte aligned base and
// rows) that lands each element in a byte of shared memory, the padded layout kind::mxf8f6f4
// reads e2m1 in: boxes of 128 elements x box_rows, 128-byte swizzle.
bool encode_e2m1_padded_2d(CUtensorMap* map, const void* base, uint64_t K, uint64_t rows,
                           uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {K, rows};
  const cuuint64_t strides[1] = {K / 2};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bsfp8_status check_common(const void* A, const void* B, const void* sa, const void* sb,
                          const int32_t* off, const int32_t* ids, void* C, int64_t M_total,
                          int N, int K, int G, int E) {
  if (!off || !B || !sb) return BSFP8_ERR_NULL;
  if (M_total > 0 && (!A || !sa || !C)) return BSFP8_ERR_NULL;
  if (M_total < 0 || M_total > INT32_MAX || N < 128 || N % 128 != 0 || K < 128 ||
      K % 128 != 0 || G < 1 || E < 1 || (int64_t)E * N > INT32_MAX)
    return BSFP8_ERR_SHAPE;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(sa, 4) ||
      !aligned(sb, 4) || !aligned(off, 4) || !aligned(ids, 4))
    return BSFP8_ERR_ALIGN;
  return BSFP8_OK;
}

// Estimated makespan of a blockwise tile configuration, in tile times: persistent CTAs (or
// CTA pairs) take tiles with a static stride, so the busiest one runs ceil(tiles / units) of
// them.  The expert offsets live on the device, so the row tiles are estimated from M_total
// and E as for an even split of the rows (E * ceil(M_total / (E * rows))).
double blockwise_makespan(int64_t M_total, int N, int E, int tile_rows, int units) {
  const double per_expert = std::ceil((double)M_total / ((double)E * tile_rows));
  const double row_tiles = (double)E * per_expert;
  const double tiles = row_tiles * (double)((N + 255) / 256);
  return std::ceil(tiles / (double)(units > 0 ? units : 1));
}

// Tile configuration for a launch.  Candidates, all with the role warps on a TMEM
// sub-partition of their own (a sub-partition that runs producer or MMA issue next to
// epilogue warps slows those warps down about twofold, so the 128-row single-CTA layouts
// lose): 96 x 256 on one CTA; 192 x 256 on a CTA pair; and 224 x 256 on an asymmetric pair,
// whose 128-row peer runs epilogue warps only.  Per tile, measured on GB300, a pair tile
// takes about 0.95 and a 224-row pair tile about 0.97 of a one-CTA 96-row tile's time.  The
// one-CTA tile is kept unless a pair form's estimated makespan is at least kSwitchMargin
// smaller (the estimates count whole waves, so an error of one tile can flip them).  The
// environment variable BSFP8_BLOCKWISE_TILE (cta1_96 | pair_192 | pair_224 | cta1_256 |
// pair_256 | pair_160 | pair_128 | cta1_128 | cta1_96x192 | pair_192x192 | cta1_128x192)
// selects a configuration.
constexpr double kPair192Time = 0.95;  // 192 x 256 pair tile time / 96 x 256 one-CTA tile time
constexpr double kPair224Time = 0.97;  // 224 x 256 pair tile time / 96 x 256 one-CTA tile time
constexpr double kSwitchMargin = 0.92;

BlockwiseTile choose_blockwise_tile(int64_t M_total, int N, int E, int num_sms) {
  if (const char* v = std::getenv("BSFP8_BLOCKWISE_TILE")) {
    if (!std::strcmp(v, "cta1_256")) return TILE_CTA1_256;
    if (!std::strcmp(v, "pair_256")) return TILE_PAIR_256;
    if (!std::strcmp(v, "pair_160")) return TILE_PAIR_160;
    if (!std::strcmp(v, "pair_128")) return TILE_PAIR_128;
    if (!std::strcmp(v, "cta1_128")) return TILE_CTA1_128;
    if (!std::strcmp(v, "cta1_96")) return TILE_CTA1_96;
    if (!std::strcmp(v, "pair_192")) return TILE_PAIR_192;
    if (!std::strcmp(v, "cta1_96x192")) return TILE_CTA1_96x192;
    if (!std::strcmp(v, "pair_192x192")) return TILE_PAIR_192x192;
    if (!std::strcmp(v, "cta1_128x192")) return TILE_CTA1_128x192;
    if (!std::strcmp(v, "pair_224")) return TILE_PAIR_224;
  }
  const double single = blockwise_makespan(M_total, N, E, 96, num_sms);
  const double pair192 = blockwise_makespan(M_total, N, E, 192, num_sms / 2) * kPair192Time;
  const double pair224 = blockwise_makespan(M_total, N, E, 224, num_sms / 2) * kPair224Time;
  const double best_pair = std::min(pair192, pair224);
  if (best_pair >= kSwitchMargin * single) return TILE_CTA1_96;
  return pair224 <= pair192 ? TILE_PAIR_224 : TILE_PAIR_192;
}

// MXFP8 kernel choice from the average token rows per expert (the per-expert counts live on
// the device).  Measured on GB300 (K = 7168, N = 2048 / 4096, L2 flushed):
//  - balanced routing favours the swap-AB tiles up to ~50 rows per expert (128 experts x
//    16-32 rows: 597 us against 692 us on the CTA-pair kernel; x 32-64 rows: 613 against
//    707) and the CTA-pair kernel from ~60 (64 experts x 48-80 rows: 373 against 404);
//  - Zipf-skewed routing favours the CTA-pair kernel already at 32 rows per expert (64
//    experts x 2048 rows: 189 us against 235; 128 x 4096: 676 against 904), its heavy
//    experts' tiles sharing each wave with the light experts' weight-streaming tiles;
//  - the split (experts with >= kMxPairMinRows rows on the CTA-pair kernel, then the others
//    on 64-row swap-AB tiles, two launches one after the other) stays near the better of the
//    two between 24 and 56 rows per expert: balanced 611 / 618 us (swap-AB 607 / 613),
//    skewed 201 / 663 / 225 us (CTA-pair 190 / 684 / 196, swap-AB 235 / 903 / 225).
// So: swap-AB up to 24 rows per expert, the split up to 56, the CTA-pair kernel above.
// BSFP8_MX_KERNEL (pair | swap | split) overrides the choice.
constexpr int64_t kMxPairMinRows = 256;
enum class MxPlan { Swap, Pair, Split };
MxPlan choose_mx_plan(int64_t M_total, int E) {
  if (const char* v = std::getenv("BSFP8_MX_KERNEL")) {
    if (!std::strcmp(v, "pair")) return MxPlan::Pair;
    if (!std::strcmp(v, "swap")) return MxPlan::Swap;
    if (!std::strcmp(v, "split")) return MxPlan::Split;
  }
  if (M_total <= (int64_t)24 * E) return MxPlan::Swap;
  if (E > 1 && M_total <= (int64_t)56 * E) return MxPlan::Split;
  return MxPlan::Pair;
}

// fp4 operands: CTA-pair tiles once the average row group no longer fits one 128-token
// swap-AB tile (measured with 8 experts, N = 4096, K = 7168: swap-AB ahead for all three
// pairs up to 128 rows per expert, the CTA pair from 192).  BSFP8_MX_KERNEL = pair | swap
// overrides (split: swap-AB, the fp4 forms having no split).
bool choose_fp4_pair(int64_t M_total, int E) {
  if (const char* v = std::getenv("BSFP8_MX_KERNEL")) {
    if (!std::strcmp(v, "pair")) return true;
    if (!std::strcmp(v, "swap") || !std::strcmp(v, "split")) return false;
  }
  return M_total > (int64_t)128 * E;
}

// Token rows per MXFP8 tile: the smallest of 32 / 64 / 128 that holds the average expert
// (decode batches give a few tokens per expert).  BSFP8_MX_TN overrides it.
int choose_mx_token_tile(int64_t M_total, int E) {
  if (const char* v = std::getenv("BSFP8_MX_TN")) {
    const int t = std::atoi(v);
    if (t == 32 || t == 64 || t == 128) return t;
  }
  const int64_t avg = (M_total + E - 1) / E;
  return avg <= 32 ? 32 : avg <= 64 ? 64 : 128;
}

}  // namespace
}  // namespace bsfp8

using namespace bsfp8;

namespace bsfp8 {
namespace {

// Grouped GEMMs over G row groups; group g multiplies the weights of expert ids[g] (of E
// experts in B), or of expert g when ids is null.
bsfp8_status blockwise_gemm(const void* A, const void* B, const float* a_scales,
                            const float* b_scales, const int32_t* offsets, const int32_t* ids,
                            void* C, int64_t M_total, int N, int K, int G, int E,
                            cudaStream_t stream) {
  bsfp8_status st = check_common(A, B, a_scales, b_scales, offsets, ids, C, M_total, N, K, G, E);
  if (st != BSFP8_OK) return st;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != BSFP8_OK) return st;
  if (M_total == 0) return BSFP8_OK;
  GemmArgs args{offsets, a_scales, b_scales, C, M_total, N, K, G, dev->err_word, ids, E, 0};
  auto run = [&](BlockwiseTile tile, const GemmArgs& a) {
    CUtensorMap tmA, tmB;
    if (!encode_u8_2d(&tmA, A, (uint64_t)K, (uint64_t)M_total, 128,
                      (uint32_t)blockwise_a_rows(tile)) ||
        !encode_u8_2d(&tmB, B, (uint64_t)K, (uint64_t)E * N, 128,
                      (uint32_t)blockwise_b_rows(tile)))
      return BSFP8_ERR_CUDA;
    return launch_bsfp8_blockwise(tile, tmA, tmB, a, dev->num_sms, stream) == cudaSuccess
               ? BSFP8_OK
               : BSFP8_ERR_CUDA;
  };
  if (const char* v = std::getenv("BSFP8_BLOCKWISE_TILE")) {
    if (!std::strcmp(v, "split")) {
      // groups of at least split_rows rows on 224-row CTA-pair tiles, then the others on
      // 96-row tiles (two launches on `stream`, each over its own groups)
      const char* r = std::getenv("BSFP8_BLOCKWISE_SPLIT_ROWS");
      const int64_t split_rows = r ? std::atoll(r) : 448;
      GemmArgs heavy = args, light = args;
      heavy.min_group_rows = split_rows;
      light.max_group_rows = split_rows;
      const bsfp8_status s1 = run(TILE_PAIR_224, heavy);
      return s1 != BSFP8_OK ? s1 : run(TILE_CTA1_96, light);
    }
  }
  return run(choose_blockwise_tile(M_total, N, G, dev->num_sms), args);
}

// packed_b: b_scales are in the 512-byte block layout of bsmxfp8_pack_b_scales (both kernels:
// a swap-AB tile's weights are one 128-row block, a CTA-pair tile's two).
bsfp8_status mx_gemm(const void* A, const void* B, const uint8_t* a_scales,
                     const uint8_t* b_scales, const int32_t* offsets, const int32_t* ids,
                     void* C, int64_t M_total, int N, int K, int G, int E, cudaStream_t stream,
                     bool packed_b = false) {
  bsfp8_status st = check_common(A, B, a_scales, b_scales, offsets, ids, C, M_total, N, K, G, E);
  if (st != BSFP8_OK) return st;
  if (packed_b && !aligned(b_scales, 16)) return BSFP8_ERR_ALIGN;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != BSFP8_OK) return st;
  if (M_total == 0) return BSFP8_OK;
  GemmArgs args{offsets, a_scales, b_scales, C, M_total, N, K, G, dev->err_word, ids, E,
                packed_b ? 1 : 0};
  const MxPlan plan = choose_mx_plan(M_total, G);
  CUtensorMap tmB;
  if (!encode_u8_2d(&tmB, B, (uint64_t)K, (uint64_t)E * N, 128, 128)) return BSFP8_ERR_CUDA;
  if (plan != MxPlan::Swap) {
    CUtensorMap tmA;
    if (!encode_u8_2d(&tmA, A, (uint64_t)K, (uint64_t)M_total, 128, 128)) return BSFP8_ERR_CUDA;
    GemmArgs heavy = args;
    if (plan == MxPlan::Split) heavy.min_group_rows = kMxPairMinRows;
    if (launch_bsmxfp8_pair(tmA, tmB, heavy, dev->num_sms, stream) != cudaSuccess)
      return BSFP8_ERR_CUDA;
    if (plan == MxPlan::Pair) return BSFP8_OK;
    args.max_group_rows = kMxPairMinRows;
  }
  // the groups below kMxPairMinRows rows under Split run 64-row token tiles (measured faster
  // than 32 or 128 rows there)
  const int tn = plan == MxPlan::Split && !std::getenv("BSFP8_MX_TN")
                     ? 64
                     : choose_mx_token_tile(M_total, G);
  CUtensorMap tmA;
  if (!encode_u8_2d(&tmA, A, (uint64_t)K, (uint64_t)M_total, 128, (uint32_t)tn))
    return BSFP8_ERR_CUDA;
  return launch_bsmxfp8(tn, tmA, tmB, args, dev->num_sms, stream) == cudaSuccess ? BSFP8_OK
                                                                                 : BSFP8_ERR_CUDA;
}

// Formats per operand.  (MXFP8, MXFP8) is mx_gemm; (MXFP4, MXFP4) and (NVFP4, NVFP4) run
// the swap-AB kernel with the fp4 MMA kinds on the packed tiles as loaded; (MXFP8, MXFP4)
// runs kind::mxf8f6f4 on e2m1 weight tiles that the tensor map loads padded.
// BSFP8_FP4_MMA=convert runs the converting kernels for every pair (the forms before the fp4
// kinds, kept for comparison).
bool fp4_mma_kind() {
  const char* v = std::getenv("BSFP8_FP4_MMA");
  return !(v && std::strcmp(v, "convert") == 0);
}

bsfp8_status mx_fmt_gemm(int a_fmt, int b_fmt, const void* A, const void* B,
                         const uint8_t* a_scales, const uint8_t* b_scales, bool packed_b,
                         const int32_t* offsets, const int32_t* ids, void* C, int64_t M_total,
                         int N, int K, int G, int E, cudaStream_t stream) {
  if (a_fmt == BSMX_MXFP8 && b_fmt == BSMX_MXFP8)
    return mx_gemm(A, B, a_scales, b_scales, offsets, ids, C, M_total, N, K, G, E, stream,
                   packed_b);
  const bool nv = a_fmt == BSMX_NVFP4 && b_fmt == BSMX_NVFP4;
  const bool a_fp4 = a_fmt == BSMX_MXFP4 || nv;
  const bool mx4 = b_fmt == BSMX_MXFP4 && (a_fmt == BSMX_MXFP8 || a_fmt == BSMX_MXFP4);
  if (!nv && !mx4) return BSFP8_ERR_FORMAT;
  if (nv && packed_b) return BSFP8_ERR_FORMAT;  // the packed block layout holds UE8M0 codes
  bsfp8_status st = check_common(A, B, a_scales, b_scales, offsets, ids, C, M_total, N, K, G, E);
  if (st != BSFP8_OK) return st;
  if (packed_b && !aligned(b_scales, 16)) return BSFP8_ERR_ALIGN;
  if (nv && (!aligned(a_scales, 8) || !aligned(b_scales, 8))) return BSFP8_ERR_ALIGN;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != BSFP8_OK) return st;
  if (M_total == 0) return BSFP8_OK;
  GemmArgs args{offsets, a_scales, b_scales, C, M_total, N, K, G, dev->err_word, ids, E,
                packed_b ? 1 : 0};
  // Prefill-sized batches (more than 128 token rows per row group on average) run the
  // CTA-pair 256 x 256 kernel on the fp4 kinds: mxfp8 x mxfp4 with its weights loaded padded
  // (32-byte aligned B), the fp4 x fp4 pairs in K blocks of 256 where the scale rows are
  // chunkable (K % 512 == 0 for mxfp4, K % 256 for nvfp4; 16-byte aligned row-major scales).
  if (fp4_mma_kind() && choose_fp4_pair(M_total, G)) {
    const int pf = a_fmt == BSMX_MXFP8 ? 1 : nv ? 3 : 2;
    const bool ok = pf == 1 ? aligned(B, 32)
                            : !packed_b && K % (nv ? 256 : 512) == 0 && aligned(a_scales, 16) &&
                                  aligned(b_scales, 16);
    if (ok) {
      CUtensorMap pA, pB;
      const bool maps =
          encode_u8_2d(&pA, A, a_fp4 ? (uint64_t)K / 2 : (uint64_t)K, (uint64_t)M_total, 128,
                       128) &&
          (pf == 1 ? encode_e2m1_padded_2d(&pB, B, (uint64_t)K, (uint64_t)E * N, 128)
                   : encode_u8_2d(&pB, B, (uint64_t)K / 2, (uint64_t)E * N, 128, 128));
      if (!maps) return BSFP8_ERR_CUDA;
      return launch_bsmx_pair_fp4(pf, pA, pB, args, dev->num_sms, stream) == cudaSuccess
                 ? BSFP8_OK
                 : BSFP8_ERR_CUDA;
    }
  }
  // Both operands fp4: the MMA kinds read the packed tiles as loaded, 256 K per stage
  // (128-byte rows, 128-byte swizzle) when every scale row's codes come in aligned 16-byte
  // chunks of whole stages, else 128 K (64-byte rows, 64-byte swizzle).
  // BSFP8_FP4_STAGE_K=128 keeps 128 K.
  const bool kind = a_fp4 && fp4_mma_kind();
  // e4m3 tokens with e2m1 weights: kind::mxf8f6f4 on weight tiles loaded padded (the map
  // needs a 32-byte aligned base), else converted on chip
  const bool mixed_kind = !a_fp4 && fp4_mma_kind() && aligned(B, 32);
  // token rows per tile: the planner's choice; the converting forms hold at most 64
  const int tn = std::min(choose_mx_token_tile(M_total, G), (kind || mixed_kind) ? 128 : 64);
  // (mxfp8 x mxfp4 with 128 token rows keeps 128-K stages: a 256-K stage of e4m3 tokens and
  // padded weights takes 64 KB, two stages only)
  const char* sk_env = std::getenv("BSFP8_FP4_STAGE_K");
  const bool wide = (kind || mixed_kind) && !(sk_env && std::strcmp(sk_env, "128") == 0) &&
                    !(mixed_kind && tn >= 128) && K % (nv ? 256 : 512) == 0 &&
                    aligned(a_scales, 16) && (packed_b || aligned(b_scales, 16));
  const uint32_t box = wide ? 128 : 64;  // bytes of packed e2m1 per row and stage
  CUtensorMap tmA, tmB;
  const bool ok_a = a_fp4 ? encode_u8_2d(&tmA, A, (uint64_t)K / 2, (uint64_t)M_total, box,
                                         (uint32_t)tn, kind)
                          : encode_u8_2d(&tmA, A, (uint64_t)K, (uint64_t)M_total, 128,
                                         (uint32_t)tn);
  const bool ok_b = mixed_kind
                        ? encode_e2m1_padded_2d(&tmB, B, (uint64_t)K, (uint64_t)E * N, 128)
                        : encode_u8_2d(&tmB, B, (uint64_t)K / 2, (uint64_t)E * N, box, 128, kind);
  if (!ok_a || !ok_b) return BSFP8_ERR_CUDA;
  const int stage_k = wide ? 256 : 128;
  const cudaError_t e =
      nv ? launch_bsnvfp4(tn, kind, stage_k, tmA, tmB, args, dev->num_sms, stream)
         : launch_bsmxfp4(tn, a_fp4, kind || mixed_kind, stage_k, tmA, tmB, args, dev->num_sms,
                          stream);
  return e == cudaSuccess ? BSFP8_OK : BSFP8_ERR_CUDA;
}

}  // namespace
}  // namespace bsfp8

extern "C" bsfp8_status bsmx_grouped_gemm(int a_format, int b_format, const void* A,
                                          const void* B, const uint8_t* a_scales,
                                          const uint8_t* b_scales, int b_scales_packed,
                                          const int32_t* group_offsets,
                                          const int32_t* expert_ids, void* C, int64_t M_total,
                                          int N, int K, int num_groups, int num_experts,
                                          cudaStream_t stream) {
  if (!expert_ids && num_groups != num_experts) return BSFP8_ERR_SHAPE;
  return mx_fmt_gemm(a_format, b_format, A, B, a_scales, b_scales, b_scales_packed != 0,
                     group_offsets, expert_ids, C, M_total, N, K, num_groups, num_experts,
                     stream);
}

extern "C" bsfp8_status bsfp8_grouped_gemm(const void* A, const void* B, const float* a_scales,
                                           const float* b_scales, const int32_t* expert_offsets,
                                           void* C, int64_t M_total, int N, int K,
                                           int num_experts, cudaStream_t stream) {
  return blockwise_gemm(A, B, a_scales, b_scales, expert_offsets, nullptr, C, M_total, N, K,
                        num_experts, num_experts, stream);
}

extern "C" bsfp8_status bsfp8_grouped_gemm_ids(const void* A, const void* B, const float* a_scales,
                                               const float* b_scales, const int32_t* group_offsets,
                                               const int32_t* expert_ids, void* C, int64_t M_total,
                                               int N, int K, int num_groups, int num_experts,
                                               cudaStream_t stream) {
  if (!expert_ids) return BSFP8_ERR_NULL;
  return blockwise_gemm(A, B, a_scales, b_scales, group_offsets, expert_ids, C, M_total, N, K,
                        num_groups, num_experts, stream);
}

extern "C" bsfp8_status bsmxfp8_grouped_gemm(const void* A, const void* B, const uint8_t* a_scales,
                                             const uint8_t* b_scales, const int32_t* expert_offsets,
                                             void* C, int64_t M_total, int N, int K,
                                             int num_experts, cudaStream_t stream) {
  return mx_gemm(A, B, a_scales, b_scales, expert_offsets, nullptr, C, M_total, N, K,
                 num_experts, num_experts, stream);
}

extern "C" bsfp8_status bsmxfp8_grouped_gemm_ids(const void* A, const void* B,
                                                 const uint8_t* a_scales, const uint8_t* b_scales,
                                                 const int32_t* group_offsets,
                                                 const int32_t* expert_ids, void* C,
                                                 int64_t M_total, int N, int K, int num_groups,
                                                 int num_experts, cudaStream_t stream) {
  if (!expert_ids) return BSFP8_ERR_NULL;
  return mx_gemm(A, B, a_scales, b_scales, group_offsets, expert_ids, C, M_total, N, K,
                 num_groups, num_experts, stream);
}

extern "C" bsfp8_status bsmxfp8_pack_b_scales(const uint8_t* b_scales, uint8_t* b_scales_packed,
                                              int num_experts, int N, int K, cudaStream_t stream) {
  if (!b_scales || !b_scales_packed) return BSFP8_ERR_NULL;
  if (num_experts < 1 || N < 128 || N % 128 != 0 || K < 128 || K % 128 != 0 ||
      (int64_t)num_experts * N > INT32_MAX)
    return BSFP8_ERR_SHAPE;
  if (!aligned(b_scales, 4) || !aligned(b_scales_packed, 16)) return BSFP8_ERR_ALIGN;
  DeviceInfo* dev = nullptr;
  bsfp8_status st = device_info(&dev);
  if (st != BSFP8_OK) return st;
  return launch_pack_mx_b_scales(b_scales, b_scales_packed, num_experts, N, K, dev->num_sms,
                                 stream) == cudaSuccess
             ? BSFP8_OK
             : BSFP8_ERR_CUDA;
}

extern "C" bsfp8_status bsmxfp8_grouped_gemm_prepacked(const void* A, const void* B,
                                                       const uint8_t* a_scales,
                                                       const uint8_t* b_scales_packed,
                                                       const int32_t* expert_offsets, void* C,
                                                       int64_t M_total, int N, int K,
                                                       int num_experts, cudaStream_t stream) {
  return mx_gemm(A, B, a_scales, b_scales_packed, expert_offsets, nullptr, C, M_total, N, K,
                 num_experts, num_experts, stream, true);
}

extern "C" bsfp8_status bsfp8_check_wait_timeout(int64_t limit_ns, cudaStream_t stream) {
  if (limit_ns <= 0 || limit_ns > 1000000000LL) return BSFP8_ERR_SHAPE;
  DeviceInfo* dev = nullptr;
  bsfp8_status st = device_info(&dev);
  if (st != BSFP8_OK) return st;
  wait_timeout_check_kernel<<<1, 32, 0, stream>>>(dev->err_word, (uint64_t)limit_ns);
  return cudaGetLastError() == cudaSuccess ? BSFP8_OK : BSFP8_ERR_CUDA;
}

extern "C" bsfp8_status bsmxfp8_tmem_plan(int block_k, int epilogue_n, int vec, int overlap,
                                          int32_t* out) {
  if (!out) return BSFP8_ERR_NULL;
  TmemPlan p;
  if (block_k == 0) {
    p = mx_pair_tmem_plan();  // the plan the CTA-pair MXFP8 kernel is compiled with
  } else {
    if (block_k < 0 || epilogue_n <= 0 || (vec != 16 && vec != 32) || block_k % vec != 0)
      return BSFP8_ERR_SHAPE;
    p = tmem_overlap_plan(block_k, epilogue_n, vec, overlap != 0);
  }
  const int32_t v[9] = {p.left_offset,    p.left_cols,    p.right_offset,
                        p.right_cols,     p.a_scale_offset, p.a_scale_cols,
                        p.b_scale_offset, p.b_scale_cols, p.early_release_subtile};
  for (int i = 0; i < 9; ++i) out[i] = v[i];
  return BSFP8_OK;
}

extern "C" bsfp8_status bsfp8_blockwise_plan(int64_t M_total, int N, int num_experts,
                                            int num_sms, int32_t* out) {
  if (!out) return BSFP8_ERR_NULL;
  if (M_total < 0 || N < 128 || N % 128 != 0 || num_experts < 1 || num_sms < 2)
    return BSFP8_ERR_SHAPE;
  const BlockwiseTile tile = choose_blockwise_tile(M_total, N, num_experts, num_sms);
  const int ctas = (tile == TILE_PAIR_256 || tile == TILE_PAIR_160 || tile == TILE_PAIR_128 ||
                    tile == TILE_PAIR_192 || tile == TILE_PAIR_192x192 ||
                    tile == TILE_PAIR_224) ? 2 : 1;
  out[0] = tile == TILE_PAIR_224 ? 224 : blockwise_a_rows(tile) * ctas;
  out[1] = blockwise_b_rows(tile) * ctas;
  out[2] = ctas;
  return BSFP8_OK;
}

extern "C" bsfp8_status bsmxfp8_plan(int64_t M_total, int num_experts, int32_t* out) {
  if (!out) return BSFP8_ERR_NULL;
  if (M_total < 0 || num_experts < 1) return BSFP8_ERR_SHAPE;
  const MxPlan plan = choose_mx_plan(M_total, num_experts);
  out[0] = plan == MxPlan::Swap ? 0 : plan == MxPlan::Pair ? 1 : 2;
  out[1] = plan == MxPlan::Pair ? 0
           : plan == MxPlan::Split && !std::getenv("BSFP8_MX_TN")
               ? 64
               : choose_mx_token_tile(M_total, num_experts);
  out[2] = plan == MxPlan::Split ? (int32_t)kMxPairMinRows : 0;
  return BSFP8_OK;
}

extern "C" bsfp8_status bsmx_plan(int64_t M_total, int num_groups, int32_t* out) {
  if (!out) return BSFP8_ERR_NULL;
  if (M_total < 0 || num_groups < 1) return BSFP8_ERR_SHAPE;
  const bool kinds = fp4_mma_kind();
  out[0] = kinds && choose_fp4_pair(M_total, num_groups) ? 1 : 0;
  out[1] = out[0] ? 0 : std::min(choose_mx_token_tile(M_total, num_groups), kinds ? 128 : 64);
  return BSFP8_OK;
}

extern "C" bsfp8_status bsfp8_get_device_error(cudaStream_t stream, int* code) {
  if (!code) return BSFP8_ERR_NULL;
  DeviceInfo* dev = nullptr;
  bsfp8_status st = device_info(&dev);
  if (st != BSFP8_OK) return st;
  int v = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess ||
      cudaMemcpyAsync(&v, dev->err_word, sizeof(int), cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaMemsetAsync(dev->err_word, 0, sizeof(int), stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return BSFP8_ERR_CUDA;
  *code = v;
  return BSFP8_OK;
}

extern "C" const char* bsfp8_status_string(bsfp8_status s) {
  switch (s) {
    case BSFP8_OK: return "ok";
    case BSFP8_ERR_NULL: return "null pointer";
    case BSFP8_ERR_SHAPE: return "invalid shape";
    case BSFP8_ERR_ALIGN: return "misaligned pointer";
    case BSFP8_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3";
    case BSFP8_ERR_CUDA: return "CUDA call failed";
    case BSFP8_ERR_DEVICE_OFFSETS: return "device: invalid expert offsets";
    case BSFP8_ERR_DEVICE_TIMEOUT: return "device: pipeline wait timed out";
    case BSFP8_ERR_DEVICE_EXPERT_IDS: return "device: expert id out of range";
    case BSFP8_ERR_FORMAT: return "unsupported operand format pair";
    case BSFP8_ERR_DEVICE_BOUNDS: return "device (debug build): tile outside the problem";
  }
  return "unknown status";
}

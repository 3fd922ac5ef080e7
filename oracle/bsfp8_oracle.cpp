// bsfp8 oracle: a plain, slow CPU statement of the blockwise-scaled FP8 grouped GEMM.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and its
// Python binding) may include, link, load or call this file.  Only the test suite,
// the smoke check and the benchmark's CPU-baseline leg use it.  It shares no code,
// header, table or constant with the CUDA kernels.
//
// What it computes (the plain definition, written out):
//
//   For every group g, every row m in [off[g], off[g+1]) and every column n < N, with
//   e = expert_ids[g] (e = g when no expert_ids are given),
//     C[m,n] = bf16_RNE( sum_kb  sa(m,kb) * sb(e,n,kb) * sum_{k in block kb} dec(A[m,k]) * dec(B[e,n,k]) )
//     T[m,n] = sum_kb |sa*sb| * sum_{k in block kb} |dec(A[m,k]) * dec(B[e,n,k])|
//
//   blockwise mode (K blocks of 128):
//     sa(m,kb)   = a_scales[kb, m]             fp32, layout [K/128, M_total]
//     sb(e,n,kb) = b_scales[e, n/128, kb]      fp32, layout [E, N/128, K/128]
//   MX mode (K blocks of 32):
//     sa(m,kb)   = 2^(a_scales[m, kb] - 127)   UE8M0, layout [M_total, K/32]
//     sb(e,n,kb) = 2^(b_scales[e, n, kb] - 127) UE8M0, layout [E, N, K/32]
//   Block-scaled formats per operand (bsfp8_oracle_fmt), as named in the Gluon example:
//     mxfp8  elements e4m3, one byte each          scale UE8M0 per 32 K
//     mxfp4  elements e2m1, two per byte along K   scale UE8M0 per 32 K
//     nvfp4  elements e2m1, two per byte along K   scale e4m3 per 16 K
//   so the term of k is dec(A[m,k]) * dec(B[e,n,k]) * sa(m, k/vec_a) * sb(e, n, k/vec_b);
//   the K blocks of the sum are min(vec_a, vec_b) wide.  A packed row holds K/2 bytes;
//   element k of a row is the low nibble of byte k/2 for even k, the high nibble for odd k.
//
// Sources:
//  * promote_accumulators (MAX kernels, linalg/grouped_matmul_sm100_blockwise_fp8),
//    description and Args: each per-K-block MMA partial is multiplied by the A scale of
//    its row and the B scale of its (expert, N block, K block) and added into fp32
//    register tiles; b_scales has shape [num_experts, N // BN, K // BK]; expert_ids maps
//    a group to its expert's rows of B; problem_shape is (M, N, K).
//  * Overlapping Accumulator Block-Scaled Matrix Multiplication (Triton Gluon example),
//    random_quantized_tensor / make_problem: the reference result of a block-scaled MMA is
//    the matmul of the dequantized operands, value * scale repeated over VEC_SIZE K
//    elements (32 for uint8 UE8M0 scales, 16 for nvfp4's float8_e4m3fn scales);
//    async_mma_scaled_impl: operands are "e4m3", or "e2m1" when stored as uint8 (two fp4
//    elements packed per byte along K); Fixed Configuration: the format pairs (mxfp8,
//    mxfp8), (mxfp8, mxfp4), (mxfp4, mxfp4), (nvfp4, nvfp4).
//
// Precision (the plain reading; every step is exact except where stated):
//  * dec() is the exact e4m3 ("fn") or e2m1 value in double.
//  * Each product dec(a)*dec(b) is exact in double (4-bit significands), and every
//    partial sum of one 128-wide block is exact too (the products span 2^-18 .. 2^18,
//    so 128 of them need < 53 bits).  nvfp4's e4m3 scales multiply exactly as well.
//  * sa*sb is exact in double (two fp32 significands).  The product with the block sum
//    and the sum over blocks round in double (relative error ~1e-16).
//  * The double result is rounded once, directly, to bf16 with round-to-nearest-even.
//
// Build: g++ -O2 -ffp-contract=off -shared -fPIC -pthread (no fast-math: the order of the
// arithmetic is the order written here).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// Encodings (OCP 8-bit floating point: E4M3 "fn" and the E8M0 scale type).
// ---------------------------------------------------------------------------

// e4m3 "fn": sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
// subnormal (M/8) * 2^-6; S.1111.111 is NaN; there is no infinity.
double e4m3_value(uint8_t code) {
  const int sign = code >> 7;
  const int E = (code >> 3) & 0xF;
  const int M = code & 0x7;
  double mag;
  if (E == 0xF && M == 0x7) return std::nan("");
  if (E == 0)
    mag = std::ldexp((double)M / 8.0, -6);
  else
    mag = std::ldexp(1.0 + (double)M / 8.0, E - 7);
  return sign ? -mag : mag;
}

// e2m1 (the 4-bit element of mxfp4 / nvfp4): sign (bit 3), 2 exponent bits (bias 1),
// 1 mantissa bit; exponent 0 is subnormal (M/2) * 2^0; no NaN, no infinity.  The
// magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6.
double e2m1_value(uint8_t nibble) {
  const int sign = (nibble >> 3) & 1;
  const int E = (nibble >> 1) & 0x3;
  const int M = nibble & 0x1;
  const double mag = (E == 0) ? (double)M / 2.0 : std::ldexp(1.0 + (double)M / 2.0, E - 1);
  return sign ? -mag : mag;
}

// UE8M0: 2^(code - 127); 0xFF is NaN.
double ue8m0_value(uint8_t code) {
  if (code == 0xFF) return std::nan("");
  return std::ldexp(1.0, (int)code - 127);
}

struct Lut {
  double e4m3[256];
  double ue8m0[256];
  double e2m1[16];
  Lut() {
    for (int c = 0; c < 256; ++c) {
      e4m3[c] = e4m3_value((uint8_t)c);
      ue8m0[c] = ue8m0_value((uint8_t)c);
    }
    for (int c = 0; c < 16; ++c) e2m1[c] = e2m1_value((uint8_t)c);
  }
};
const Lut& lut() {
  static const Lut table;
  return table;
}

// Round a double once, directly, to bf16 (1 sign, 8 exponent, 7 mantissa bits) with
// round-to-nearest, ties-to-even.  Quantum of the binade 2^E is 2^(E-7) for E >= -126 and
// 2^-133 below (subnormals).  Magnitudes that round to 2^128 or more become infinity.
uint16_t bf16_rne(double x) {
  if (std::isnan(x)) return 0x7FC0;
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  const double a = std::fabs(x);
  if (a == 0.0) return sign;
  if (std::isinf(a)) return sign | 0x7F80;
  int e2;
  std::frexp(a, &e2);      // a = f * 2^e2, f in [0.5, 1)  ->  floor(log2 a) = e2 - 1
  int E = e2 - 1;
  if (E < -126) E = -126;
  const double quantum = std::ldexp(1.0, E - 7);
  const double r = std::nearbyint(a / quantum);  // a / quantum is exact; default mode = RNE
  const double v = r * quantum;                   // exact
  if (v >= std::ldexp(1.0, 128)) return sign | 0x7F80;
  const float f = (float)v;  // exact: v has at most 8 significant bits and is in fp32 range
  uint32_t bits;
  std::memcpy(&bits, &f, 4);
  return sign | (uint16_t)(bits >> 16);
}

enum Mode { BLOCKWISE = 0, MX = 1 };

// Block-scaled operand formats (MX mode).
enum Format { MXFP8 = 0, MXFP4 = 1, NVFP4 = 2 };

struct Problem {
  Mode mode;
  const uint8_t* A;          // [M_total, K]
  const uint8_t* B;          // [E, N, K]
  const void* a_scales;      // see header comment
  const void* b_scales;
  const int32_t* offsets;    // [E+1]
  int64_t M_total;
  int64_t N, K;
  int64_t E;                 // groups (row segments)
  const int32_t* expert_ids; // [E] group -> expert of B, or nullptr (group g uses expert g)
  int64_t num_experts;       // experts in B and b_scales
  Format a_fmt = MXFP8;      // MX mode only
  Format b_fmt = MXFP8;
};

bool packed(Format f) { return f != MXFP8; }
int64_t vec_of(Format f) { return f == NVFP4 ? 16 : 32; }
int64_t row_bytes(Format f, int64_t K) { return packed(f) ? K / 2 : K; }

// Element k of an operand row in format f.
double elem(const Lut& L, Format f, const uint8_t* row, int64_t k) {
  if (!packed(f)) return L.e4m3[row[k]];
  const uint8_t byte = row[k / 2];
  return L.e2m1[(k & 1) ? (byte >> 4) : (byte & 0xF)];
}

// Scale code c of a block in format f.
double scale_of(const Lut& L, Format f, uint8_t c) { return f == NVFP4 ? L.e4m3[c] : L.ue8m0[c]; }

int check(const Problem& p) {
  if (p.M_total < 0 || p.N <= 0 || p.K <= 0 || p.E <= 0) return 2;
  const int64_t blk = (p.mode == BLOCKWISE) ? 128 : 32;
  if (p.K % blk != 0) return 2;
  if (p.mode == MX && (p.a_fmt < MXFP8 || p.a_fmt > NVFP4 || p.b_fmt < MXFP8 || p.b_fmt > NVFP4))
    return 2;
  if (p.mode == BLOCKWISE && p.N % 128 != 0) return 2;
  if (p.offsets[0] != 0 || p.offsets[p.E] != p.M_total) return 6;
  for (int64_t e = 0; e < p.E; ++e)
    if (p.offsets[e + 1] < p.offsets[e]) return 6;
  if (p.num_experts <= 0) return 2;
  if (p.expert_ids) {
    for (int64_t g = 0; g < p.E; ++g)
      if (p.expert_ids[g] < 0 || p.expert_ids[g] >= p.num_experts) return 8;
  } else if (p.num_experts != p.E) {
    return 2;
  }
  return 0;
}

// Group that owns row m: the g with off[g] <= m < off[g+1] (empty groups own no row).
int64_t group_of_row(const Problem& p, int64_t m) {
  int64_t lo = 0, hi = p.E - 1;
  while (lo < hi) {  // smallest e with off[e+1] > m
    const int64_t mid = (lo + hi) / 2;
    if (p.offsets[mid + 1] > m) hi = mid; else lo = mid + 1;
  }
  return lo;
}

// One output element of an MX problem with per-operand formats: K blocks of
// min(vec_a, vec_b) elements, each block's exact sum times its two scales.
void element_fmt(const Problem& p, const Lut& L, int64_t m, int64_t n, int64_t e,
                 uint16_t* c_out, double* t_out) {
  const int64_t va = vec_of(p.a_fmt), vb = vec_of(p.b_fmt);
  const int64_t blk = std::min(va, vb);
  const uint8_t* arow = p.A + m * row_bytes(p.a_fmt, p.K);
  const uint8_t* brow = p.B + (e * p.N + n) * row_bytes(p.b_fmt, p.K);
  const uint8_t* asc = (const uint8_t*)p.a_scales + m * (p.K / va);
  const uint8_t* bsc = (const uint8_t*)p.b_scales + (e * p.N + n) * (p.K / vb);
  double acc = 0.0, tsum = 0.0;
  for (int64_t k0 = 0; k0 < p.K; k0 += blk) {
    double inner = 0.0, inner_abs = 0.0;
    for (int64_t k = k0; k < k0 + blk; ++k) {
      const double prod = elem(L, p.a_fmt, arow, k) * elem(L, p.b_fmt, brow, k);
      inner += prod;
      inner_abs += std::fabs(prod);
    }
    const double s = scale_of(L, p.a_fmt, asc[k0 / va]) * scale_of(L, p.b_fmt, bsc[k0 / vb]);
    acc += s * inner;
    tsum += std::fabs(s) * inner_abs;
  }
  *c_out = bf16_rne(acc);
  if (t_out) *t_out = tsum;
}

// One output element, straight from the definition above.
void element(const Problem& p, int64_t m, int64_t n, uint16_t* c_out, double* t_out) {
  const Lut& L = lut();
  // expert_ids: "mapping from group index to expert row offset in B" (promote_accumulators)
  const int64_t g = group_of_row(p, m);
  const int64_t e = p.expert_ids ? (int64_t)p.expert_ids[g] : g;
  if (p.mode == MX && (p.a_fmt != MXFP8 || p.b_fmt != MXFP8)) {
    element_fmt(p, L, m, n, e, c_out, t_out);
    return;
  }
  const int64_t blk = (p.mode == BLOCKWISE) ? 128 : 32;
  const int64_t nkb = p.K / blk;
  const uint8_t* arow = p.A + m * p.K;
  const uint8_t* brow = p.B + (e * p.N + n) * p.K;
  double acc = 0.0, tsum = 0.0;
  for (int64_t kb = 0; kb < nkb; ++kb) {
    double inner = 0.0, inner_abs = 0.0;
    for (int64_t k = kb * blk; k < (kb + 1) * blk; ++k) {
      const double prod = L.e4m3[arow[k]] * L.e4m3[brow[k]];
      inner += prod;
      inner_abs += std::fabs(prod);
    }
    double sa, sb;
    if (p.mode == BLOCKWISE) {
      sa = (double)((const float*)p.a_scales)[kb * p.M_total + m];
      sb = (double)((const float*)p.b_scales)[(e * (p.N / 128) + n / 128) * nkb + kb];
    } else {
      sa = L.ue8m0[((const uint8_t*)p.a_scales)[m * nkb + kb]];
      sb = L.ue8m0[((const uint8_t*)p.b_scales)[(e * p.N + n) * nkb + kb]];
    }
    const double s = sa * sb;
    acc += s * inner;
    tsum += std::fabs(s) * inner_abs;
  }
  *c_out = bf16_rne(acc);
  if (t_out) *t_out = tsum;
}

int resolve_threads(int nthreads) {
  if (nthreads > 0) return nthreads;
  const unsigned hc = std::thread::hardware_concurrency();
  return hc ? (int)hc : 1;
}

// Full output: rows split into contiguous chunks, one per thread.
int run_full(const Problem& p, uint16_t* C, double* T, int nthreads) {
  const int rc = check(p);
  if (rc) return rc;
  const int nt = resolve_threads(nthreads);
  auto work = [&](int64_t r0, int64_t r1) {
    for (int64_t m = r0; m < r1; ++m)
      for (int64_t n = 0; n < p.N; ++n)
        element(p, m, n, C + m * p.N + n, T ? T + m * p.N + n : nullptr);
  };
  std::vector<std::thread> pool;
  const int64_t chunk = (p.M_total + nt - 1) / nt;
  for (int t = 0; t < nt; ++t) {
    const int64_t r0 = t * chunk, r1 = std::min<int64_t>(p.M_total, r0 + chunk);
    if (r0 >= r1) break;
    pool.emplace_back(work, r0, r1);
  }
  for (auto& th : pool) th.join();
  return 0;
}

// Sampled output: the elements (rows[i], cols[i]) only.
int run_points(const Problem& p, const int64_t* rows, const int64_t* cols, int64_t npts,
               uint16_t* C, double* T, int nthreads) {
  const int rc = check(p);
  if (rc) return rc;
  for (int64_t i = 0; i < npts; ++i)
    if (rows[i] < 0 || rows[i] >= p.M_total || cols[i] < 0 || cols[i] >= p.N) return 2;
  const int nt = resolve_threads(nthreads);
  auto work = [&](int64_t i0, int64_t i1) {
    for (int64_t i = i0; i < i1; ++i)
      element(p, rows[i], cols[i], C + i, T ? T + i : nullptr);
  };
  std::vector<std::thread> pool;
  const int64_t chunk = (npts + nt - 1) / nt;
  for (int t = 0; t < nt; ++t) {
    const int64_t i0 = t * chunk, i1 = std::min<int64_t>(npts, i0 + chunk);
    if (i0 >= i1) break;
    pool.emplace_back(work, i0, i1);
  }
  for (auto& th : pool) th.join();
  return 0;
}

}  // namespace

extern "C" {

// Return codes: 0 ok, 2 bad shape, 6 bad expert offsets, 8 expert id out of range (same
// meaning as the library's).

double bsfp8_oracle_e4m3_decode(uint8_t code) { return lut().e4m3[code]; }
double bsfp8_oracle_ue8m0_decode(uint8_t code) { return lut().ue8m0[code]; }
uint16_t bsfp8_oracle_bf16_rne(double x) { return bf16_rne(x); }

int bsfp8_oracle_blockwise(const uint8_t* A, const uint8_t* B, const float* a_scales,
                           const float* b_scales, const int32_t* offsets, int64_t M_total,
                           int64_t N, int64_t K, int64_t E, uint16_t* C, double* T,
                           int nthreads) {
  Problem p{BLOCKWISE, A, B, a_scales, b_scales, offsets, M_total, N, K, E, nullptr, E};
  return run_full(p, C, T, nthreads);
}

int bsfp8_oracle_mx(const uint8_t* A, const uint8_t* B, const uint8_t* a_scales,
                    const uint8_t* b_scales, const int32_t* offsets, int64_t M_total,
                    int64_t N, int64_t K, int64_t E, uint16_t* C, double* T, int nthreads) {
  Problem p{MX, A, B, a_scales, b_scales, offsets, M_total, N, K, E, nullptr, E};
  return run_full(p, C, T, nthreads);
}

int bsfp8_oracle_blockwise_points(const uint8_t* A, const uint8_t* B, const float* a_scales,
                                  const float* b_scales, const int32_t* offsets,
                                  int64_t M_total, int64_t N, int64_t K, int64_t E,
                                  const int64_t* rows, const int64_t* cols, int64_t npts,
                                  uint16_t* C, double* T, int nthreads) {
  Problem p{BLOCKWISE, A, B, a_scales, b_scales, offsets, M_total, N, K, E, nullptr, E};
  return run_points(p, rows, cols, npts, C, T, nthreads);
}

int bsfp8_oracle_mx_points(const uint8_t* A, const uint8_t* B, const uint8_t* a_scales,
                           const uint8_t* b_scales, const int32_t* offsets, int64_t M_total,
                           int64_t N, int64_t K, int64_t E, const int64_t* rows,
                           const int64_t* cols, int64_t npts, uint16_t* C, double* T,
                           int nthreads) {
  Problem p{MX, A, B, a_scales, b_scales, offsets, M_total, N, K, E, nullptr, E};
  return run_points(p, rows, cols, npts, C, T, nthreads);
}

// Grouped GEMM with an expert indirection: G groups of rows (offsets [G+1]), group g using
// expert expert_ids[g] of num_experts (B [num_experts, N, K] and its scales).  mode 0 is
// blockwise (fp32 scales), 1 is MX (UE8M0 scales).
int bsfp8_oracle_ids(int mode, const uint8_t* A, const uint8_t* B, const void* a_scales,
                     const void* b_scales, const int32_t* offsets, const int32_t* expert_ids,
                     int64_t M_total, int64_t N, int64_t K, int64_t G, int64_t num_experts,
                     uint16_t* C, double* T, int nthreads) {
  if (!expert_ids || (mode != 0 && mode != 1)) return 2;
  Problem p{mode == 0 ? BLOCKWISE : MX, A, B, a_scales, b_scales, offsets, M_total, N, K, G,
            expert_ids, num_experts};
  return run_full(p, C, T, nthreads);
}

// MX grouped GEMM with a format per operand (0 mxfp8, 1 mxfp4, 2 nvfp4): A [M_total,
// K or K/2 bytes], a_scales [M_total, K/vec_a]; B [num_experts, N, K or K/2 bytes],
// b_scales [num_experts, N, K/vec_b]; G groups of rows (offsets [G+1]); group g uses expert
// expert_ids[g], or expert g when expert_ids is null (then num_experts must equal G).
int bsfp8_oracle_fmt(int a_fmt, int b_fmt, const uint8_t* A, const uint8_t* B,
                     const uint8_t* a_scales, const uint8_t* b_scales, const int32_t* offsets,
                     const int32_t* expert_ids, int64_t M_total, int64_t N, int64_t K, int64_t G,
                     int64_t num_experts, uint16_t* C, double* T, int nthreads) {
  Problem p{MX, A, B, a_scales, b_scales, offsets, M_total, N, K, G, expert_ids, num_experts,
            (Format)a_fmt, (Format)b_fmt};
  return run_full(p, C, T, nthreads);
}

int bsfp8_oracle_fmt_points(int a_fmt, int b_fmt, const uint8_t* A, const uint8_t* B,
                            const uint8_t* a_scales, const uint8_t* b_scales,
                            const int32_t* offsets, const int32_t* expert_ids, int64_t M_total,
                            int64_t N, int64_t K, int64_t G, int64_t num_experts,
                            const int64_t* rows, const int64_t* cols, int64_t npts, uint16_t* C,
                            double* T, int nthreads) {
  Problem p{MX, A, B, a_scales, b_scales, offsets, M_total, N, K, G, expert_ids, num_experts,
            (Format)a_fmt, (Format)b_fmt};
  return run_points(p, rows, cols, npts, C, T, nthreads);
}

double bsfp8_oracle_e2m1_decode(uint8_t nibble) { return lut().e2m1[nibble & 0xF]; }

int bsfp8_oracle_threads(int nthreads) { return resolve_threads(nthreads); }

}  // extern "C"

// Seeded synthetic inputs for the blockwise-scaled FP8 grouped GEMM.
//
// This module makes inputs only.  It holds none of the GEMM's arithmetic: no decode of
// the stored bytes, no products, no sums.  Both the oracle and the CUDA library consume
// its outputs; neither is linked into it and it is linked into neither.
//
// Every value is a pure function of (seed, stream, element index), so the bytes do not
// depend on the thread count and are the same on x86-64 and AArch64: the only floating
// point operations are IEEE basic operations and sqrt, compiled with -ffp-contract=off,
// and the logarithm/exponential used below are written out here instead of taken from
// the platform libm.
//
// Recipe (stated in the library's design notes):
//  * N(0,1) source values: Marsaglia's polar method on counter-based uniforms.
//  * Blockwise FP8: scale = amax/448 in fp32 per 1x128 block of A and per 128x128 block
//    of B (amax 0 -> scale 1); code = e4m3(x / scale), x/scale in fp32, round to nearest
//    even, saturating at +-448.
//  * MXFP8: per 1x32 block, scale = 2^ceil(log2(amax/448)) with amax/448 in fp32 and the
//    ceiling taken from its bits; UE8M0 code = exponent + 127 (amax 0 -> 127);
//    code = e4m3(x * 2^-exponent), saturating.
//  * Exact-arithmetic inputs: values on the e2m1 grid {0, 0.5, 1, 1.5, 2, 3, 4, 6} with a
//    random sign, stored as e4m3; scales drawn from {0.5, 1, 2} (UE8M0 126..128).  The
//    fp4-grid-values-with-power-of-two-scales idea is random_quantized_tensor in the
//    Triton Gluon example "Overlapping Accumulator Block-Scaled Matrix Multiplication".
//  * Routing: uniform multinomial; Zipf(s) over a seeded permutation of experts; uniform
//    integer token counts per expert.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// Counter-based random numbers (splitmix64 finaliser, Steele/Lea/Flood 2014).
// ---------------------------------------------------------------------------
inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(seed * 0x9E3779B97F4A7C15ull + stream * 0xD1B54A32D192ED03ull + 1);
}
inline uint64_t hash_k(uint64_t key, uint64_t ctr) { return mix64(key ^ mix64(ctr + 0x632BE59BD9B4E019ull)); }
inline uint64_t hash3(uint64_t seed, uint64_t stream, uint64_t ctr) {
  return hash_k(stream_key(seed, stream), ctr);
}
// Uniform in [0, 1) with 53 random bits.
inline double unit(uint64_t h) { return (double)(h >> 11) * (1.0 / 9007199254740992.0); }

// Natural logarithm for x > 0 (finite), from frexp and the atanh series
// ln(m) = 2*t*(1 + t^2/3 + ... + t^18/19), t = (m-1)/(m+1), m in [sqrt(1/2), sqrt(2)].
double my_log(double x) {
  int e;
  double m = std::frexp(x, &e);  // x = m * 2^e, m in [0.5, 1)
  m *= 2.0;
  e -= 1;                        // m in [1, 2)
  if (m > 1.4142135623730951) {
    m *= 0.5;
    e += 1;
  }
  const double t = (m - 1.0) / (m + 1.0);
  const double t2 = t * t;
  // Horner form of 1 + t2/3 + t2^2/5 + ... + t2^9/19 (coefficients rounded to double)
  static const double inv_odd[10] = {1.0,        1.0 / 3.0,  1.0 / 5.0,  1.0 / 7.0,
                                     1.0 / 9.0,  1.0 / 11.0, 1.0 / 13.0, 1.0 / 15.0,
                                     1.0 / 17.0, 1.0 / 19.0};
  double poly = inv_odd[9];
  for (int i = 8; i >= 0; --i) poly = poly * t2 + inv_odd[i];
  return 2.0 * t * poly + (double)e * 0.6931471805599453;
}

// exp(x) for |x| < 700: x = n*ln2 + r, |r| <= ln2/2, Taylor series of exp(r) to 24 terms.
double my_exp(double x) {
  const double n = std::nearbyint(x / 0.6931471805599453);
  const double r = x - n * 0.6931471805599453;
  double term = 1.0, sum = 1.0;
  for (int k = 1; k <= 24; ++k) {
    term *= r / (double)k;
    sum += term;
  }
  return std::ldexp(sum, (int)n);
}

// Pair j of standard normals for (seed, stream): Marsaglia's polar method, trying up to
// 64 counter values; the chance of 64 rejections is ~1e-43.
inline void normal_pair(uint64_t key, uint64_t j, double* z0, double* z1) {
  for (uint64_t t = 0; t < 64; ++t) {
    const uint64_t h1 = hash_k(key, (j << 7) | (2 * t));
    const uint64_t h2 = hash_k(key, (j << 7) | (2 * t + 1));
    const double x = 2.0 * unit(h1) - 1.0;
    const double y = 2.0 * unit(h2) - 1.0;
    const double s = x * x + y * y;
    if (s > 0.0 && s < 1.0) {
      const double f = std::sqrt(-2.0 * my_log(s) / s);
      *z0 = x * f;
      *z1 = y * f;
      return;
    }
  }
  *z0 = 0.0;
  *z1 = 0.0;
}

// count fp32 normals for element indices [start, start+count); start and count even.
void normals(uint64_t seed, uint64_t stream, uint64_t start, uint64_t count, float* out) {
  const uint64_t key = stream_key(seed, stream);
  for (uint64_t i = 0; i < count; i += 2) {
    double z0, z1;
    normal_pair(key, (start + i) >> 1, &z0, &z1);
    out[i] = (float)z0;
    out[i + 1] = (float)z1;
  }
}

// ---------------------------------------------------------------------------
// fp32 -> e4m3 ("fn"), round to nearest even, saturating to +-448.
// ---------------------------------------------------------------------------
uint8_t e4m3_encode(float xf) {
  if (std::isnan(xf)) return 0x7F;
  const uint8_t sign = std::signbit(xf) ? 0x80 : 0x00;
  const double a = std::fabs((double)xf);
  if (a >= 448.0) return sign | 0x7E;
  if (a == 0.0) return sign;
  int E;
  double q;  // quantum of a's binade
  if (a < 0.015625) {  // below 2^-6: subnormal quantum 2^-9
    E = -6;
    q = 0.001953125;
  } else {
    int e2;
    std::frexp(a, &e2);
    E = e2 - 1;  // a in [2^E, 2^(E+1))
    q = std::ldexp(1.0, E - 3);
  }
  double r = std::rint(a / q);  // a / q is exact; default rounding = nearest even
  if (a < 0.015625) {
    // subnormal: value r * 2^-9, r in [0, 8]; r == 8 is 2^-6, the smallest normal.
    if (r >= 8.0) return sign | 0x08;
    return sign | (uint8_t)r;
  }
  // normal: value r * 2^(E-3), r in [8, 16]
  if (r >= 16.0) {
    r = 8.0;
    E += 1;
  }
  if (E > 8 || (E == 8 && r > 14.0)) return sign | 0x7E;  // above 448 (cannot happen)
  return sign | (uint8_t)(((E + 7) << 3) | ((int)r - 8));
}

// ceil(log2(r)) for a positive finite fp32 r, from its exponent and significand.
int ceil_log2(float r) {
  int e2;
  const float f = std::frexp(r, &e2);  // r = f * 2^e2, f in [0.5, 1)
  return (f == 0.5f) ? e2 - 1 : e2;
}

// ---------------------------------------------------------------------------
// Threading helper: run fn(i) for i in [0, n) on nt threads, static chunks.
// ---------------------------------------------------------------------------
template <class F>
void parallel_for(int64_t n, int nthreads, F fn) {
  int nt = nthreads > 0 ? nthreads : (int)std::max(1u, std::thread::hardware_concurrency());
  if (nt > n) nt = (int)std::max<int64_t>(1, n);
  if (nt <= 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  std::vector<std::thread> pool;
  const int64_t chunk = (n + nt - 1) / nt;
  for (int t = 0; t < nt; ++t) {
    const int64_t i0 = t * chunk, i1 = std::min<int64_t>(n, i0 + chunk);
    if (i0 >= i1) break;
    pool.emplace_back([=, &fn]() {
      for (int64_t i = i0; i < i1; ++i) fn(i);
    });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// Streams used by the Python front end (any distinct values work).
//   1: A source values   2: B source values   3: routing   4: outlier rows
//   5: A exact values    6: B exact values    7: A exact scales   8: B exact scales

void bsfp8_gen_normals(uint64_t seed, uint64_t stream, uint64_t start, uint64_t count,
                       float* out) {
  // any start/count: generate the covering even range into a scratch buffer
  const uint64_t s0 = start & ~1ull;
  const uint64_t s1 = (start + count + 1) & ~1ull;
  std::vector<float> tmp(s1 - s0);
  normals(seed, stream, s0, s1 - s0, tmp.data());
  std::memcpy(out, tmp.data() + (start - s0), count * sizeof(float));
}

uint8_t bsfp8_gen_e4m3_encode(float x) { return e4m3_encode(x); }
int bsfp8_gen_ceil_log2(float r) { return ceil_log2(r); }
double bsfp8_gen_log(double x) { return my_log(x); }
double bsfp8_gen_exp(double x) { return my_exp(x); }

// Rows of a [rows, K] operand, sourced from N(0,1) (row r uses element indices
// (r0 + r) * K + k), optional per-row multiplier, quantized per 1 x 128 block.
// Q: [rows, K] e4m3 codes.  scales: fp32 laid out [K/128, scale_ld] with this operand's
// rows at columns [0, rows) (scale_ld >= rows), i.e. scales[kb * scale_ld + r].
void bsfp8_gen_blockwise_rows(uint64_t seed, uint64_t stream, int64_t r0, int64_t rows,
                              int64_t K, const float* row_mult, uint8_t* Q, float* scales,
                              int64_t scale_ld, int nthreads) {
  const int64_t nkb = K / 128;
  parallel_for(rows, nthreads, [&](int64_t r) {
    float x[128];
    const float mult = row_mult ? row_mult[r] : 1.0f;
    for (int64_t kb = 0; kb < nkb; ++kb) {
      normals(seed, stream, (uint64_t)((r0 + r) * K + kb * 128), 128, x);
      float amax = 0.0f;
      for (int i = 0; i < 128; ++i) {
        x[i] *= mult;
        amax = std::max(amax, std::fabs(x[i]));
      }
      const float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
      for (int i = 0; i < 128; ++i) Q[r * K + kb * 128 + i] = e4m3_encode(x[i] / s);
      scales[kb * scale_ld + r] = s;
    }
  });
}

// B operand [E, N, K] from N(0,1) (row e*N+n uses element indices (e*N+n)*K + k),
// quantized per 128 x 128 block; scales [E, N/128, K/128].
void bsfp8_gen_blockwise_b(uint64_t seed, uint64_t stream, int64_t E, int64_t N, int64_t K,
                           uint8_t* Q, float* scales, int nthreads) {
  const int64_t nnb = N / 128, nkb = K / 128;
  parallel_for(E * nnb * nkb, nthreads, [&](int64_t blk) {
    const int64_t kb = blk % nkb, nb = (blk / nkb) % nnb, e = blk / (nkb * nnb);
    std::vector<float> x(128 * 128);
    float amax = 0.0f;
    for (int i = 0; i < 128; ++i) {
      const int64_t row = e * N + nb * 128 + i;
      normals(seed, stream, (uint64_t)(row * K + kb * 128), 128, &x[i * 128]);
      for (int j = 0; j < 128; ++j) amax = std::max(amax, std::fabs(x[i * 128 + j]));
    }
    const float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
    for (int i = 0; i < 128; ++i) {
      const int64_t row = e * N + nb * 128 + i;
      for (int j = 0; j < 128; ++j) Q[row * K + kb * 128 + j] = e4m3_encode(x[i * 128 + j] / s);
    }
    scales[(e * nnb + nb) * nkb + kb] = s;
  });
}

// MXFP8 rows: [rows, K] from N(0,1) (row r uses element indices (r0 + r) * K + k),
// optional per-row multiplier, quantized per 1 x 32 block with UE8M0 scales
// [rows, K/32] (row-major).
void bsfp8_gen_mx_rows(uint64_t seed, uint64_t stream, int64_t r0, int64_t rows, int64_t K,
                       const float* row_mult, uint8_t* Q, uint8_t* scales, int nthreads) {
  const int64_t nsb = K / 32;
  parallel_for(rows, nthreads, [&](int64_t r) {
    float x[32];
    const float mult = row_mult ? row_mult[r] : 1.0f;
    for (int64_t sb = 0; sb < nsb; ++sb) {
      normals(seed, stream, (uint64_t)((r0 + r) * K + sb * 32), 32, x);
      float amax = 0.0f;
      for (int i = 0; i < 32; ++i) {
        x[i] *= mult;
        amax = std::max(amax, std::fabs(x[i]));
      }
      int e = 0;
      if (amax > 0.0f) {
        e = ceil_log2(amax / 448.0f);
        e = std::min(127, std::max(-127, e));
      }
      for (int i = 0; i < 32; ++i) Q[r * K + sb * 32 + i] = e4m3_encode(std::ldexp(x[i], -e));
      scales[r * nsb + sb] = (uint8_t)(e + 127);
    }
  });
}

// Exact-arithmetic operand: count codes, each a value of the e2m1 grid
// {0, 0.5, 1, 1.5, 2, 3, 4, 6} with a random sign, stored as e4m3.
void bsfp8_gen_exact_codes(uint64_t seed, uint64_t stream, int64_t count, uint8_t* Q,
                           int nthreads) {
  static const float grid[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
  const int64_t per = 4096;
  parallel_for((count + per - 1) / per, nthreads, [&](int64_t c) {
    for (int64_t i = c * per; i < std::min(count, (c + 1) * per); ++i) {
      const uint64_t h = hash3(seed, stream, (uint64_t)i);
      const float v = grid[h & 7];
      Q[i] = e4m3_encode(((h >> 3) & 1) ? -v : v);
    }
  });
}

// Exact-arithmetic scales: fp32 in {0.5, 1, 2} (or UE8M0 codes 126..128).
void bsfp8_gen_exact_scales_f32(uint64_t seed, uint64_t stream, int64_t count, float* s) {
  static const float v[3] = {0.5f, 1.0f, 2.0f};
  for (int64_t i = 0; i < count; ++i) s[i] = v[hash3(seed, stream, (uint64_t)i) % 3];
}
void bsfp8_gen_exact_scales_ue8m0(uint64_t seed, uint64_t stream, int64_t count, uint8_t* s) {
  for (int64_t i = 0; i < count; ++i) s[i] = (uint8_t)(126 + hash3(seed, stream, (uint64_t)i) % 3);
}

// fp4 operand as random_quantized_tensor draws it: every e2m1 code (4 bits, sign
// included) uniform, two per byte along K (element 2i in the low nibble of byte i).
void bsfp8_gen_fp4_bytes(uint64_t seed, uint64_t stream, int64_t nbytes, uint8_t* out,
                         int nthreads) {
  const int64_t per = 4096;
  parallel_for((nbytes + per - 1) / per, nthreads, [&](int64_t c) {
    for (int64_t i = c * per; i < std::min(nbytes, (c + 1) * per); ++i)
      out[i] = (uint8_t)(hash3(seed, stream, (uint64_t)i) & 0xFF);
  });
}

// Power-of-two scales 2^j, j uniform in [-7, 1] (the [1/128, 2] range of
// random_quantized_tensor), as UE8M0 codes (e4m3 == 0) or as e4m3 codes (e4m3 != 0; exact:
// 2^-7 is the e4m3 subnormal 4/8 * 2^-6).
void bsfp8_gen_pow2_scales(uint64_t seed, uint64_t stream, int64_t count, int e4m3,
                           uint8_t* out, int nthreads) {
  uint8_t code[9];
  for (int j = -7; j <= 1; ++j) code[j + 7] = e4m3 ? e4m3_encode(std::ldexp(1.0f, j)) : (uint8_t)(127 + j);
  const int64_t per = 4096;
  parallel_for((count + per - 1) / per, nthreads, [&](int64_t c) {
    for (int64_t i = c * per; i < std::min(count, (c + 1) * per); ++i)
      out[i] = code[hash3(seed, stream, (uint64_t)i) % 9];
  });
}

// General positive e4m3 scale codes, uniform over the codes lo .. hi (finite, > 0).
void bsfp8_gen_e4m3_scale_codes(uint64_t seed, uint64_t stream, int64_t count, int lo, int hi,
                                uint8_t* out, int nthreads) {
  const int64_t per = 4096;
  parallel_for((count + per - 1) / per, nthreads, [&](int64_t c) {
    for (int64_t i = c * per; i < std::min(count, (c + 1) * per); ++i)
      out[i] = (uint8_t)(lo + (int)(hash3(seed, stream, (uint64_t)i) % (uint64_t)(hi - lo + 1)));
  });
}

// Routing: counts[E] of rows per expert.
// Uniform multinomial: each of M_total tokens picks expert floor(u * E).
void bsfp8_gen_route_uniform(uint64_t seed, int64_t M_total, int64_t E, int32_t* counts) {
  for (int64_t e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t t = 0; t < M_total; ++t) {
    int64_t e = (int64_t)(unit(hash3(seed, 3, (uint64_t)t)) * (double)E);
    if (e >= E) e = E - 1;
    counts[e] += 1;
  }
}

// Zipf(s): expert perm[r-1] gets weight r^-s (rank r = 1..E, perm a seeded shuffle);
// each token draws an expert from these weights.  Then the zero_lowest experts of
// lowest weight are emptied and their rows moved to the expert of rank 1.
void bsfp8_gen_route_zipf(uint64_t seed, int64_t M_total, int64_t E, double s,
                          int64_t zero_lowest, int32_t* counts) {
  std::vector<int64_t> perm(E);
  for (int64_t i = 0; i < E; ++i) perm[i] = i;
  for (int64_t i = E - 1; i > 0; --i) {  // Fisher-Yates
    const int64_t j = (int64_t)(unit(hash3(seed, 9, (uint64_t)i)) * (double)(i + 1));
    std::swap(perm[i], perm[std::min(j, i)]);
  }
  std::vector<double> cdf(E);
  double tot = 0.0;
  for (int64_t r = 0; r < E; ++r) {
    tot += my_exp(-s * my_log((double)(r + 1)));
    cdf[r] = tot;
  }
  for (int64_t e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t t = 0; t < M_total; ++t) {
    const double u = unit(hash3(seed, 3, (uint64_t)t)) * tot;
    int64_t r = (int64_t)(std::upper_bound(cdf.begin(), cdf.end(), u) - cdf.begin());
    if (r >= E) r = E - 1;
    counts[perm[r]] += 1;
  }
  for (int64_t z = 0; z < zero_lowest && z < E - 1; ++z) {
    const int64_t victim = perm[E - 1 - z];
    counts[perm[0]] += counts[victim];
    counts[victim] = 0;
  }
}

// Uniform integer rows per expert in [lo, hi].
void bsfp8_gen_route_counts(uint64_t seed, int64_t E, int64_t lo, int64_t hi, int32_t* counts) {
  for (int64_t e = 0; e < E; ++e) {
    int64_t c = lo + (int64_t)(unit(hash3(seed, 3, (uint64_t)e)) * (double)(hi - lo + 1));
    if (c > hi) c = hi;
    counts[e] = (int32_t)c;
  }
}

// Outlier rows: the n_out rows with the smallest hash values (ties by index) get mask 1.
void bsfp8_gen_outlier_rows(uint64_t seed, int64_t M_total, int64_t n_out, uint8_t* mask) {
  std::vector<std::pair<uint64_t, int64_t>> h(M_total);
  for (int64_t m = 0; m < M_total; ++m) h[m] = {hash3(seed, 4, (uint64_t)m), m};
  n_out = std::min(n_out, M_total);
  std::partial_sort(h.begin(), h.begin() + n_out, h.end());
  for (int64_t m = 0; m < M_total; ++m) mask[m] = 0;
  for (int64_t i = 0; i < n_out; ++i) mask[h[i].second] = 1;
}

}  // extern "C"

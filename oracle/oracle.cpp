/*
 * oracle.cpp -- plain, slow, obviously correct CPU oracle for the W4A16
 * group-affine quantized matmul.  TEST INFRASTRUCTURE ONLY: only tests/,
 * the package's smoke check and the benchmark's cpu_baseline leg load it.
 * It shares no code, header or helper with the CUDA path.
 *
 * Citations (page titles; sections in quotes):
 *   [W2D2] tiny-llm book, "Week 2 Day 2: Keep W4 Packed"
 *   [G4MK] "Gemma 4 E4B & E2B -- single-launch Metal megakernels + lossless
 *          speculative decoding" (RESMP-DEV model card)
 *   [HY4]  "Hy4-preview Metal kernels for llama.cpp"
 *
 * What it computes (all in fp64, every step exact except the final sum):
 *   q[n,k] = (Wq[n][k/8] >> 4*(k%8)) & 0xF        [W2D2 "Packed Storage Layout"]
 *   w[n,k] = q[n,k] * s[n,k/G] + b[n,k/G]         [W2D2 "Reconstruct a Stored Group",
 *                                                   equation w^ = q s + b]
 *   y[m,n] = sum_k x[m,k] * w[n,k]                [W2D2 "Mathematical Formulation",
 *                                                   C[i,k] = sum_j A[i,j] B[k,j]]
 * with G = 64 [G4MK "Usage": the dequant path assumes group size 64], or
 * G = 128 through the _g entry points [W2D2 "Packed Storage Layout": the
 * book's group size; its "Reconstruct a Stored Group" is the same equation
 * with 128 codes per scale and bias].  The
 * loops follow [W2D2 "Computation Flow"]: for every output, walk groups g,
 * packs p inside the group and the eight nibbles of each pack, reconstruct
 * the weight and add a*w to one accumulator.  The pages accumulate in float;
 * this oracle uses one fp64 accumulator ([HY4 "Results": a float64 reference])
 * so its own rounding is far below any tolerance.  It also returns
 * sum_k |x*w| per output, which the acceptance bound uses.
 *
 * Letters: the page writes C = A B^T with A (M x N) and the reduction over
 * its N.  Here x[M][K], Wq[N][K/8], y[M][N], reduction over K.
 *
 * mm_id (routed experts): y[t,n] = sum_k x[t,k] * w_{ids[t]}[n,k] for T
 * tokens with one expert id each; an id outside 0..E-1 gives a zero row.
 * The pages name llama.cpp's mul_mat_id ([HY4] kernel table) without a
 * signature; top-1 routing is the plainest reading.
 *
 * STQ1_0 (the ternary format of [HY4]): stq1_* below, with the block layout
 * and the reading of the lane decode written beside the code.  Activations
 * are float32 and outputs fp64, as in the page's _f32 kernels.
 *
 * bf16: raw 16-bit patterns.  Decoding and round-to-nearest-even encoding are
 * written here from the bfloat16 definition (1 sign, 8 exponent bits with
 * bias 127, 7 fraction bits; subnormal spacing 2^-133), with plain fp64
 * arithmetic -- no bit tricks shared with any other code.
 */
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

const int kGroup = 64;

// ---- bfloat16 from its definition -------------------------------------------

double bf16_decode(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int efield = (h >> 7) & 0xFF;
  const int frac = h & 0x7F;
  double mag;
  if (efield == 0xFF) {
    if (frac != 0) return std::nan("");
    mag = INFINITY;
  } else if (efield == 0) {
    mag = std::ldexp((double)frac, -133);                 // subnormal: frac * 2^-126 * 2^-7
  } else {
    mag = std::ldexp((double)(128 + frac), efield - 127 - 7);  // 1.frac * 2^(e-127)
  }
  return sign ? -mag : mag;
}

// Nearest bf16 to v, ties to the even significand; NaN -> quiet NaN with v's
// sign; magnitudes that round to 2^128 or beyond -> infinity.
uint16_t bf16_encode(double v) {
  const uint16_t sign = std::signbit(v) ? 0x8000 : 0;
  if (std::isnan(v)) return (uint16_t)(sign | 0x7FC0);
  double a = std::fabs(v);
  if (std::isinf(a)) return (uint16_t)(sign | 0x7F80);
  if (a == 0.0) return sign;
  int ex;
  std::frexp(a, &ex);          // a = f * 2^ex, f in [0.5, 1): binade exponent is ex - 1
  int e = ex - 1;
  int spacing_exp = (e < -126) ? -133 : e - 7;
  double qv = std::ldexp(a, -spacing_exp);  // exact: a scaled by a power of two
  double fl = std::floor(qv);
  double diff = qv - fl;       // exact
  double r;
  if (diff > 0.5) r = fl + 1.0;
  else if (diff < 0.5) r = fl;
  else r = (std::fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
  double res = std::ldexp(r, spacing_exp);
  if (res >= std::ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
  if (res < std::ldexp(1.0, -126)) {
    // subnormal (r < 128) or exactly the smallest normal (r == 128): the
    // integer r is then the bit pattern itself.
    return (uint16_t)(sign | (uint16_t)r);
  }
  std::frexp(res, &ex);
  e = ex - 1;
  double sig = std::ldexp(res, -(e - 7));   // in [128, 256)
  return (uint16_t)(sign | (uint16_t)((e + 127) << 7) | (uint16_t)((int)sig - 128));
}

// ---- the definition ---------------------------------------------------------

inline int code_at(const uint32_t* Wq, int64_t K, int64_t n, int64_t k) {
  uint32_t word = Wq[n * (K / 8) + k / 8];
  return (int)((word >> (4 * (k % 8))) & 0xFu);
}

// One output element, in the page's loop order, groups of G codes.
void dot_one(const uint16_t* xrow, const uint32_t* Wq, const uint16_t* S, const uint16_t* B,
             int64_t K, int64_t n, int64_t G, double* y, double* absdot) {
  const int64_t groups = K / G;
  const int64_t words_per_group = G / 8;
  double sum = 0.0, abs_sum = 0.0;
  for (int64_t g = 0; g < groups; ++g) {
    const double scale = bf16_decode(S[n * groups + g]);
    const double bias = bf16_decode(B[n * groups + g]);
    for (int64_t p = 0; p < words_per_group; ++p) {
      const uint32_t packed = Wq[n * (K / 8) + g * words_per_group + p];
      for (int bit_offset = 0; bit_offset < 32; bit_offset += 4) {
        const int q = (int)((packed >> bit_offset) & 0xFu);
        const double w = (double)q * scale + bias;
        const double a = bf16_decode(xrow[g * G + p * 8 + bit_offset / 4]);
        sum += a * w;
        abs_sum += std::fabs(a * w);
      }
    }
  }
  *y = sum;
  if (absdot) *absdot = abs_sum;
}

template <class F>
void parallel_over(int64_t n, int threads, F fn) {
  if (threads <= 0) threads = (int)std::max(1u, std::thread::hardware_concurrency());
  if (threads > n) threads = (int)std::max<int64_t>(1, n);
  if (threads <= 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  std::vector<std::thread> pool;
  for (int t = 0; t < threads; ++t)
    pool.emplace_back([=]() {
      for (int64_t i = t; i < n; i += threads) fn(i);
    });
  for (auto& th : pool) th.join();
}

bool group_ok(int64_t G) { return G == 64 || G == 128; }
bool shape_ok(int64_t K, int64_t G = kGroup) { return group_ok(G) && K > 0 && K % G == 0; }

// ---- STQ1_0: the ternary format of [HY4] ------------------------------------
//
// One block holds 256 weights in 42 bytes [HY4 "Notes and gotchas": "42-byte
// block stride" and the block-layout note]: 32 bytes of 4-bit group codes,
// 8 bytes of group sign bits, and an fp16 scale d, in that order (the order
// the page lists them; read as the byte layout).  Weight w of a block belongs
// to group g = (w/64)*16 + w%16 at lane p = (w%64)/16 [same note].  Code
// nibble g is qs[g/2] >> 4*(g%2) (low nibble first, as the W4 codes of
// [W2D2 "Packed Storage Layout"]); sign bit g is bit g%8 of sign[g/8]; d is
// little endian.  The lane values of a group [HY4 "Results", the fourth
// decode pass]: the code's high two bits name the zero lane, its low two
// bits flip the signs of two of the other three lanes, and the sign bit
// negates the whole group.  Which two lanes the flips reach is not written
// out; the reading taken here is: the three non-zero lanes in ascending lane
// order, bit 0 flips the first, bit 1 the second, the third stays +1.
// A weight is d * v with v in {-1, 0, +1}.

const int kStqWeights = 256;
const int kStqBytes = 42;

// IEEE binary16 from its definition: 1 sign, 5 exponent bits with bias 15,
// 10 fraction bits; subnormals frac * 2^-24.
double fp16_decode(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int efield = (h >> 10) & 0x1F;
  const int frac = h & 0x3FF;
  double mag;
  if (efield == 0x1F) {
    if (frac != 0) return std::nan("");
    mag = INFINITY;
  } else if (efield == 0) {
    mag = std::ldexp((double)frac, -24);
  } else {
    mag = std::ldexp((double)(1024 + frac), efield - 15 - 10);
  }
  return sign ? -mag : mag;
}

// The four lane values of code c (0..15) under group sign s (0 or 1).
void stq1_lanes(int c, int s, int v[4]) {
  const int zero_lane = c >> 2;
  int rank = 0;  // position among the non-zero lanes, ascending
  for (int l = 0; l < 4; ++l) {
    if (l == zero_lane) {
      v[l] = 0;
      continue;
    }
    const int flip = rank == 0 ? (c & 1) : rank == 1 ? ((c >> 1) & 1) : 0;
    v[l] = flip ? -1 : 1;
    ++rank;
  }
  if (s)
    for (int l = 0; l < 4; ++l) v[l] = -v[l];
}

// Weight w (0..255) of one block.
double stq1_weight(const uint8_t* block, int w) {
  const int g = (w / 64) * 16 + w % 16;
  const int p = (w % 64) / 16;
  const int c = (block[g / 2] >> (4 * (g % 2))) & 0xF;
  const int s = (block[32 + g / 8] >> (g % 8)) & 1;
  int v[4];
  stq1_lanes(c, s, v);
  const uint16_t dbits = (uint16_t)(block[40] | (block[41] << 8));
  return fp16_decode(dbits) * (double)v[p];
}

// One output of y = x W^T: row n of a [N][K/256][42] block matrix against a
// float32 activation row, in fp64, weights in storage order.
void stq1_dot_one(const float* xrow, const uint8_t* blocks, int64_t K, int64_t n, double* y, double* absdot) {
  const int64_t nb = K / kStqWeights;
  double sum = 0.0, abs_sum = 0.0;
  for (int64_t b = 0; b < nb; ++b) {
    const uint8_t* block = blocks + (n * nb + b) * kStqBytes;
    for (int w = 0; w < kStqWeights; ++w) {
      const double a = (double)xrow[b * kStqWeights + w];
      const double wt = stq1_weight(block, w);
      sum += a * wt;
      abs_sum += std::fabs(a * wt);
    }
  }
  *y = sum;
  if (absdot) *absdot = abs_sum;
}

bool stq1_shape_ok(int64_t K) { return K > 0 && K % kStqWeights == 0; }

}  // namespace

extern "C" {

int oracle_group_size(void) { return kGroup; }

double oracle_bf16_to_double(uint16_t h) { return bf16_decode(h); }
uint16_t oracle_bf16_from_double(double v) { return bf16_encode(v); }

void oracle_bf16_from_double_array(const double* v, int64_t n, uint16_t* out, int threads) {
  const int64_t chunk = 1 << 16;
  parallel_over((n + chunk - 1) / chunk, threads, [&](int64_t c) {
    int64_t hi = std::min(n, (c + 1) * chunk);
    for (int64_t i = c * chunk; i < hi; ++i) out[i] = bf16_encode(v[i]);
  });
}

void oracle_bf16_from_float_array(const float* v, int64_t n, uint16_t* out, int threads) {
  const int64_t chunk = 1 << 16;
  parallel_over((n + chunk - 1) / chunk, threads, [&](int64_t c) {
    int64_t hi = std::min(n, (c + 1) * chunk);
    for (int64_t i = c * chunk; i < hi; ++i) out[i] = bf16_encode((double)v[i]);
  });
}

// Unit of last place of the bf16 grid at v: 2^(floor(log2|v|) - 7) for
// |v| >= 2^-126, else the subnormal spacing 2^-133.
double oracle_ulp_bf16(double v) {
  double a = std::fabs(v);
  if (a < std::ldexp(1.0, -126)) return std::ldexp(1.0, -133);
  int ex;
  std::frexp(a, &ex);
  return std::ldexp(1.0, ex - 1 - 7);
}

void oracle_bf16_to_double_array(const uint16_t* h, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_decode(h[i]);
}

void oracle_ulp_bf16_array(const double* v, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_ulp_bf16(v[i]);
}

// q[n][k] for the whole matrix.
int oracle_unpack(const uint32_t* Wq, int64_t N, int64_t K, uint8_t* q) {
  if (!Wq || !q) return -1;
  if (N < 0 || K <= 0 || K % 8) return -2;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) q[n * K + k] = (uint8_t)code_at(Wq, K, n, k);
  return 0;
}

// w[n][k] = q*s + b in fp64 for the whole matrix, groups of G codes.
int oracle_dequant_g(const uint32_t* Wq, const uint16_t* S, const uint16_t* B, int64_t N, int64_t K, int64_t G,
                     double* w) {
  if (!Wq || !S || !B || !w) return -1;
  if (N < 0 || !shape_ok(K, G)) return -2;
  const int64_t groups = K / G;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k)
      w[n * K + k] = (double)code_at(Wq, K, n, k) * bf16_decode(S[n * groups + k / G]) +
                     bf16_decode(B[n * groups + k / G]);
  return 0;
}

int oracle_dequant(const uint32_t* Wq, const uint16_t* S, const uint16_t* B, int64_t N, int64_t K,
                   double* w) {
  return oracle_dequant_g(Wq, S, B, N, K, kGroup, w);
}

// y[m][j] = sum_k x[m,k] w[cols[j], k] for j < ncols (all n when cols is NULL,
// then ncols must equal N), groups of G codes.  absdot (optional) gets
// sum_k |x w|.
int oracle_mm_g(const uint16_t* x, const uint32_t* Wq, const uint16_t* S, const uint16_t* B, int64_t M,
                int64_t N, int64_t K, int64_t G, const int64_t* cols, int64_t ncols, double* y, double* absdot,
                int threads) {
  if (!x || !Wq || !S || !B || !y) return -1;
  if (M < 0 || N < 0 || ncols < 0 || !shape_ok(K, G)) return -2;
  if (!cols && ncols != N) return -2;
  for (int64_t j = 0; cols && j < ncols; ++j)
    if (cols[j] < 0 || cols[j] >= N) return -2;
  parallel_over(ncols, threads, [&](int64_t j) {
    const int64_t n = cols ? cols[j] : j;
    for (int64_t m = 0; m < M; ++m)
      dot_one(x + m * K, Wq, S, B, K, n, G, &y[m * ncols + j], absdot ? &absdot[m * ncols + j] : nullptr);
  });
  return 0;
}

int oracle_mm(const uint16_t* x, const uint32_t* Wq, const uint16_t* S, const uint16_t* B, int64_t M,
              int64_t N, int64_t K, const int64_t* cols, int64_t ncols, double* y, double* absdot,
              int threads) {
  return oracle_mm_g(x, Wq, S, B, M, N, K, kGroup, cols, ncols, y, absdot, threads);
}

// Routed experts: Wq[E][N][K/8], S/B[E][N][K/64], ids[T]; y[t][j] for the
// sampled output columns (all N when cols is NULL).
int oracle_mm_id(const uint16_t* x, const uint32_t* Wq, const uint16_t* S, const uint16_t* B,
                 const int32_t* ids, int64_t T, int64_t N, int64_t K, int64_t E, const int64_t* cols,
                 int64_t ncols, double* y, double* absdot, int threads) {
  if (!x || !Wq || !S || !B || !ids || !y) return -1;
  if (T < 0 || N < 0 || E <= 0 || ncols < 0 || !shape_ok(K)) return -2;
  if (!cols && ncols != N) return -2;
  for (int64_t j = 0; cols && j < ncols; ++j)
    if (cols[j] < 0 || cols[j] >= N) return -2;
  const int64_t words = N * (K / 8), params = N * (K / kGroup);
  parallel_over(ncols, threads, [&](int64_t j) {
    const int64_t n = cols ? cols[j] : j;
    for (int64_t t = 0; t < T; ++t) {
      const int64_t e = ids[t];
      if (e < 0 || e >= E) {
        y[t * ncols + j] = 0.0;
        if (absdot) absdot[t * ncols + j] = 0.0;
        continue;
      }
      dot_one(x + t * K, Wq + e * words, S + e * params, B + e * params, K, n, kGroup, &y[t * ncols + j],
              absdot ? &absdot[t * ncols + j] : nullptr);
    }
  });
  return 0;
}

// ---- STQ1_0 [HY4] ---------------------------------------------------------------

double oracle_fp16_to_double(uint16_t h) { return fp16_decode(h); }

// v[4] of code c under sign s (the lane values of one group).
int oracle_stq1_lanes(int c, int s, int* v) {
  if (!v || c < 0 || c > 15 || (s != 0 && s != 1)) return -2;
  stq1_lanes(c, s, v);
  return 0;
}

// w[n][k] in fp64 for a [N][K/256][42] block matrix.
int oracle_stq1_dequant(const uint8_t* blocks, int64_t N, int64_t K, double* w) {
  if (!blocks || !w) return -1;
  if (N < 0 || !stq1_shape_ok(K)) return -2;
  const int64_t nb = K / kStqWeights;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k)
      w[n * K + k] = stq1_weight(blocks + (n * nb + k / kStqWeights) * kStqBytes, (int)(k % kStqWeights));
  return 0;
}

// y[m][j] = sum_k x[m,k] w[cols[j], k] (all n when cols is NULL), x float32.
int oracle_stq1_mm(const float* x, const uint8_t* blocks, int64_t M, int64_t N, int64_t K, const int64_t* cols,
                   int64_t ncols, double* y, double* absdot, int threads) {
  if (!x || !blocks || !y) return -1;
  if (M < 0 || N < 0 || ncols < 0 || !stq1_shape_ok(K)) return -2;
  if (!cols && ncols != N) return -2;
  for (int64_t j = 0; cols && j < ncols; ++j)
    if (cols[j] < 0 || cols[j] >= N) return -2;
  parallel_over(ncols, threads, [&](int64_t j) {
    const int64_t n = cols ? cols[j] : j;
    for (int64_t m = 0; m < M; ++m)
      stq1_dot_one(x + m * K, blocks, K, n, &y[m * ncols + j], absdot ? &absdot[m * ncols + j] : nullptr);
  });
  return 0;
}

// Routed experts over blocks[E][N][K/256][42]: y[t] = W[ids[t]] x[t]; an id
// outside 0..E-1 gives a zero row.
int oracle_stq1_mm_id(const float* x, const uint8_t* blocks, const int32_t* ids, int64_t T, int64_t N, int64_t K,
                      int64_t E, const int64_t* cols, int64_t ncols, double* y, double* absdot, int threads) {
  if (!x || !blocks || !ids || !y) return -1;
  if (T < 0 || N < 0 || E <= 0 || ncols < 0 || !stq1_shape_ok(K)) return -2;
  if (!cols && ncols != N) return -2;
  for (int64_t j = 0; cols && j < ncols; ++j)
    if (cols[j] < 0 || cols[j] >= N) return -2;
  const int64_t per_expert = N * (K / kStqWeights) * kStqBytes;
  parallel_over(ncols, threads, [&](int64_t j) {
    const int64_t n = cols ? cols[j] : j;
    for (int64_t t = 0; t < T; ++t) {
      const int64_t e = ids[t];
      if (e < 0 || e >= E) {
        y[t * ncols + j] = 0.0;
        if (absdot) absdot[t * ncols + j] = 0.0;
        continue;
      }
      stq1_dot_one(x + t * K, blocks + e * per_expert, K, n, &y[t * ncols + j],
                   absdot ? &absdot[t * ncols + j] : nullptr);
    }
  });
  return 0;
}

}  // extern "C"

// prefill.cu -- W4A16 for many activation rows (prefill; the default above 32) on the
// fifth-generation tensor cores: tcgen05.mma from shared memory into tensor
// memory (TMEM).
//
// Citations (page titles; sections in quotes):
//   [W2D2] tiny-llm book, "Week 2 Day 2: Keep W4 Packed"
//   [G4MK] "Gemma 4 E4B & E2B -- single-launch Metal megakernels + lossless
//          speculative decoding" (RESMP-DEV model card)
//   [HY4]  "Hy4-preview Metal kernels for llama.cpp"
//
// With tens of activation rows the dequantised weight tile is reused enough
// for the matmul to become a dense contraction ([W2D2] "GPU Dispatch" sends
// such batches to a separate schedule; [HY4] "Results" gives prefill its
// own loader).  This kernel expands each 64-code group of a 128-row weight
// tile ONCE into bf16 (128 + q, exact) in shared memory and multiplies it
// with up to 128 activation rows per tcgen05.mma, so the unpack work is paid
// once per weight instead of once per eight rows.
//
// It computes the canonical arithmetic of the skinny kernels (tc.cu): for
// every output row n, activation row m and 64-group g of a canonical slice,
//     acc = sum_k x_k (128 + q_k)   (four K = 16 MMA steps, fp32)
//     sx  = sum_k x_k               (four m16n8k16 MMA steps with A = 1.0)
//     p   = fma(s, acc, p);  p = fma(b - 128 s, sx, p)
// and y = bf16(((p_0 + p_1) + p_2) + ...) over the slices of tc_shape(N, K).
// The K order of the four MMA steps of a group is the skinny kernels' (each
// step sums the same sixteen codes: step 2cb + h takes codes 32cb + 8t + 2h
// + {0, 1, 4, 5}, t = 0..3), so the weight tile and the activation tile are
// both stored in that order: the codes by the unpack (one LOP3 per pair,
// as in tc.cu), the activations by a 4x4 word transpose after their TMA
// load.
//
// CTA: 15 warps, one 128-row tile x NC activation rows (NC = 32, 64, 128;
// blockIdx.y takes the next NC rows), the whole K range.  The copies run
// ahead in rings: two stages of codes (8 groups each), 5-12 activation
// tiles, four expanded weight tiles.
//   warps 0 .. NC/8 - 1   epilogue: accumulator -> registers (warp w reads
//                TMEM lanes 32 (w % 4) .. and 32 columns), the group sums from
//                MMA row 127, the per-group rescale into p, slice sums folded
//                in slice order in TMEM, bf16 stores
//   next 8 warps expansion, up to 4-6 groups ahead: rows 0-126 of the
//                weight tile as bf16 128 + q, row 127 ones, and the
//                activation tile permuted in place
//   next warp    TMA producer: per 8 groups the codes (two 128-byte-wide
//                boxes of 128 rows) and the scales and biases (128 rows x
//                16 B each); per group the activation tile (NC rows x 128 B)
//   last warp    tensor-memory allocation; lane 0 issues the MMAs of each
//                group into one of several TMEM accumulators and commits them
// Every wait is bounded: one that gives up raises W4A16_DEVICE_TIMEOUT, all
// roles leave their loops, outstanding copies and MMAs are waited for (also
// bounded) and the tensor memory is freed before the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace w4a16 {
namespace {

using namespace ptx;

constexpr int kPRows = 128;                  // rows of the MMA (the M of tcgen05.mma)
constexpr int kTileN = 127;                  // weight rows per CTA; MMA row 127 is all ones
constexpr int kATile = kPRows * 128;         // 16 KB: 128 rows x 64 bf16
constexpr int kCodeBox = kPRows * 128;       // 16 KB: 128 rows x 32 packed words (4 groups)
constexpr int kParamTile = 2 * kPRows * 16;  // scales | biases of 8 groups
constexpr uint32_t kOnesBf16x2 = 0x3F803F80u;

template <int NC>
struct PGeo {
  static constexpr int kX = NC * 128;                // activation tile: NC rows x 64 bf16
  static constexpr int kSlots = NC == 128 ? 5 : NC == 64 ? 6 : 11;  // activation tiles in flight
  static constexpr int kPSlots = 4;                  // stages of scales and biases
  static constexpr int kASlots = NC == 128 ? 4 : 6;  // expanded weight tiles
  static constexpr int kCW = 32;                     // columns per epilogue warp
  static constexpr int kEpi = NC / 8;                // epilogue warps: NC / 32 per TMEM lane quarter
  static constexpr int kThreads = 32 * (kEpi + 10);  // + 8 expansion warps, the producer, the MMA issuer
  static constexpr int kAcc = NC == 128 ? 3 : NC == 64 ? 6 : 12;  // TMEM accumulators
  static constexpr uint32_t kTmemCols = 512;         // kAcc accumulators + the slice sums
  // barriers: raw_full, raw_free per activation slot; a_full, a_free per
  // tile; acc_full, acc_free per accumulator; params full / free per
  // params stage; then two each of codes full / free
  static constexpr int kBars = 2 * kSlots + 2 * kASlots + 2 * kAcc + 2 * kPSlots + 4;
  static constexpr int kSmem = kASlots * kATile + 2 * 2 * kCodeBox + kSlots * kX + kPSlots * kParamTile +
                               kAcc * NC * 4 + kBars * 8 + 16 + 1024;
  static_assert(kSmem <= 227 * 1024, "a CTA's shared memory");
};

struct PrefillMaps {
  CUtensorMap codes;   // u32 [N][K/8], box 32 words x 128 rows, 128-byte swizzle
  CUtensorMap x;       // bf16 [M][K], box 64 x NC rows, 128-byte swizzle
  CUtensorMap scales;  // bf16 [N][K/64], box 8 groups x 128 rows
  CUtensorMap biases;
};

struct PrefillParams {
  uint16_t* y;
  int* flags;
  int N, K, M;
  int groups;  // K / 64
  int gps;     // groups per canonical slice (a multiple of 8)
};

// Logical 16-byte chunk c of row r of a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128(uint32_t tile, int r, int c) {
  return tile + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint16_t bf16_rne_bits(float v) { return f32_to_bf16_bits(v); }

// Named barrier of the `count` threads of one epilogue column quarter.
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

template <int NC>
__global__ void __launch_bounds__(PGeo<NC>::kThreads, 1) tc_prefill_kernel(const __grid_constant__ PrefillMaps maps,
                                                                  PrefillParams p) {
  using G = PGeo<NC>;
  constexpr int S = G::kSlots, AS = G::kASlots, CW = G::kCW, NB = G::kAcc, PS = G::kPSlots, EW = G::kEpi;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // layout: expanded weight tiles [AS] | codes of a stage [2][2 boxes] | activation tiles [S]
  //         | params [PS][scales | biases] | sx [NB][NC] fp32 | barriers | tmem base, abort
  const uint32_t codes0 = sb + AS * kATile;
  const uint32_t slots0 = codes0 + 2 * 2 * kCodeBox;
  const uint32_t params0 = slots0 + S * G::kX;
  const uint32_t sx0 = params0 + PS * kParamTile;
  const uint32_t bars = sx0 + NB * NC * 4;
  auto A_of = [&](int a) { return sb + (uint32_t)(a * kATile); };
  auto C_of = [&](int cs) { return codes0 + (uint32_t)(cs * 2 * kCodeBox); };
  auto X_of = [&](int s) { return slots0 + (uint32_t)(s * G::kX); };
  auto raw_full = [&](int s) { return bars + 8u * s; };               // activation tile landed (TMA)
  auto raw_free = [&](int s) { return bars + 8u * (S + s); };         // MMAs done with it
  auto a_full = [&](int a) { return bars + 8u * (2 * S + a); };       // tile expanded, activations permuted
  auto a_free = [&](int a) { return bars + 8u * (2 * S + AS + a); };  // MMAs done with the tile
  auto acc_full = [&](int b) { return bars + 8u * (2 * S + 2 * AS + b); };       // MMA commit
  auto acc_free = [&](int b) { return bars + 8u * (2 * S + 2 * AS + NB + b); };  // epilogue warps
  auto par_full = [&](int b) { return bars + 8u * (2 * S + 2 * AS + 2 * NB + b); };        // TMA
  auto par_free = [&](int b) { return bars + 8u * (2 * S + 2 * AS + 2 * NB + PS + b); };   // epilogue warps
  // two-deep: 2 codes full, 3 codes free
  auto bar2 = [&](int k, int b) { return bars + 8u * (2 * S + 2 * AS + 2 * NB + 2 * PS + 2 * (k - 2) + b); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(base + (bars - sb) + 8 * G::kBars);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(raw_full(s), 1);
      mbar_init(raw_free(s), 1);
    }
    for (int a = 0; a < AS; ++a) {
      mbar_init(a_full(a), 8);
      mbar_init(a_free(a), 1);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_free(b), EW);
    }
    for (int b = 0; b < PS; ++b) {
      mbar_init(par_full(b), 1);
      mbar_init(par_free(b), EW);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar2(2, b), 1);
      mbar_init(bar2(3, b), 8);
    }
    *s_abort = 0;
    fence_barrier_init();
  }
  const int W_EXP = EW, W_PROD = EW + 8, W_MMA = EW + 9;  // first expansion warp, producer, MMA issuer
  if (warp == W_MMA) {
    tmem_alloc(smem_u32(s_tmem), G::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *s_tmem;
  const int row0 = blockIdx.x * kTileN, col0 = blockIdx.y * NC;
  const int ng = p.groups;
  auto timeout = [&]() {
    atomicOr(p.flags, W4A16_DEVICE_TIMEOUT);
    *s_abort = 1;
  };
  // warp-uniform bounded wait (false after a timeout; a role whose partner
  // gave up times out in turn at its next wait)
  auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
    const bool ok = __all_sync(0xffffffffu, mbar_wait_parked(bar, parity));
    if (!ok && lane == 0) timeout();
    return ok;
  };
  int issued = 0, mma_done = 0;  // producer / MMA lane 0: groups requested / committed

  if (warp == W_PROD) {
    // ---- TMA producer ----
    if (lane == 0) {
      const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();
      int g = 0;
      for (; g < ng && !*s_abort; ++g) {
        const int s = g % S;
        if (g >= S && !mbar_wait_parked(raw_free(s), ((g / S) - 1) & 1)) {
          timeout();
          break;
        }
        if ((g & 7) == 0) {
          const int st = g >> 3, cs = st & 1, ps = st % PS;
          if ((st >= PS && !mbar_wait_parked(par_free(ps), ((st / PS) - 1) & 1)) ||
              (st >= 2 && !mbar_wait_parked(bar2(3, cs), ((st >> 1) - 1) & 1))) {
            timeout();
            break;
          }
          mbar_expect_tx(par_full(ps), kParamTile);
          tma_load_2d(params0 + ps * kParamTile, &maps.scales, 8 * st, row0, par_full(ps), pol_keep);
          tma_load_2d(params0 + ps * kParamTile + kParamTile / 2, &maps.biases, 8 * st, row0, par_full(ps), pol_keep);
          // the stage's codes: two 128-byte-wide boxes of four groups each
          mbar_expect_tx(bar2(2, cs), 2 * kCodeBox);
          tma_load_2d(C_of(cs), &maps.codes, 64 * st, row0, bar2(2, cs), pol_stream);
          tma_load_2d(C_of(cs) + kCodeBox, &maps.codes, 64 * st + 32, row0, bar2(2, cs), pol_stream);
        }
        mbar_expect_tx(raw_full(s), G::kX);
        tma_load_2d(X_of(s), &maps.x, 64 * g, col0, raw_full(s), pol_keep);
      }
      issued = g;
    }
  } else if (warp == W_MMA) {
    // ---- MMA issuer: accumulator b = A(g) * X(g)^T over the group's four K steps ----
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(kPRows, NC);
      int g = 0;
      for (; g < ng && !*s_abort; ++g) {
        const int s = g % S, a = g % AS, b = g % NB;
        if (!mbar_wait_parked(a_full(a), (g / AS) & 1) || (g >= NB && !mbar_wait_parked(acc_free(b), ((g / NB) - 1) & 1))) {
          timeout();
          break;
        }
        tc_fence_after_sync();
        const uint64_t ad = umma_desc_sw128(A_of(a)), bd = umma_desc_sw128(X_of(s));
#pragma unroll
        for (int j = 0; j < 4; ++j) umma_bf16(tmem + (uint32_t)(b * NC), ad + 2 * j, bd + 2 * j, idesc, j > 0);
        umma_commit(acc_full(b));
        umma_commit(a_free(a));
        umma_commit(raw_free(s));
      }
      mma_done = g;
    }
  } else if (warp >= W_EXP) {
    // ---- expansion (8 warps), up to AS groups ahead: rows 0-126 the
    // codes as bf16 128 + q, row 127 ones (its MMA row is the group sums),
    // and the activation tile permuted, both in the MMA steps' K order ----
    const int et = threadIdx.x - 32 * W_EXP;  // 0..255
    const int rr = et & 127, cb = et >> 7;
    for (int g = 0; g < ng; ++g) {
      const int s = g % S, a = g % AS, st = g >> 3, gi = g & 7, cs = st & 1;
      if (gi == 0 && !wait_all(bar2(2, cs), (st >> 1) & 1)) break;
      if (!wait_all(raw_full(s), (g / S) & 1)) break;
      if (g >= AS && !wait_all(a_free(a), ((g / AS) - 1) & 1)) break;
      const uint32_t A = A_of(a), X = X_of(s), C = C_of(cs) + (uint32_t)((gi >> 2) * kCodeBox);
      // activation tasks (row m, half xb): 2 NC / 8 consecutive rows per warp
      // (consecutive rows fall in different swizzle phases: no bank conflicts)
      constexpr int XPW = 2 * NC / 8;
      const int xtask = (warp - W_EXP) * XPW + lane;
      const bool xt = lane < XPW;
      const int m = xtask % NC, xb = xtask / NC;
      // all loads first, then the stores
      const uint4 wv = lds128(sw128(C, rr, 2 * (gi & 3) + cb));
      uint4 c[4];
      if (xt) {
#pragma unroll
        for (int t = 0; t < 4; ++t) c[t] = lds128(sw128(X, m, 4 * xb + t));
      }
      if (rr < kTileN) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          sts128(sw128(A, rr, 4 * cb + e), codes_as_bf16x2(wv.x >> (4 * e)), codes_as_bf16x2(wv.y >> (4 * e)),
                 codes_as_bf16x2(wv.z >> (4 * e)), codes_as_bf16x2(wv.w >> (4 * e)));
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) sts128(sw128(A, rr, 4 * cb + e), kOnesBf16x2, kOnesBf16x2, kOnesBf16x2, kOnesBf16x2);
      }
      if (xt) {
        sts128(sw128(X, m, 4 * xb + 0), prmt(c[0].x, c[0].z, 0x5410), prmt(c[1].x, c[1].z, 0x5410),
               prmt(c[2].x, c[2].z, 0x5410), prmt(c[3].x, c[3].z, 0x5410));
        sts128(sw128(X, m, 4 * xb + 1), prmt(c[0].x, c[0].z, 0x7632), prmt(c[1].x, c[1].z, 0x7632),
               prmt(c[2].x, c[2].z, 0x7632), prmt(c[3].x, c[3].z, 0x7632));
        sts128(sw128(X, m, 4 * xb + 2), prmt(c[0].y, c[0].w, 0x5410), prmt(c[1].y, c[1].w, 0x5410),
               prmt(c[2].y, c[2].w, 0x5410), prmt(c[3].y, c[3].w, 0x5410));
        sts128(sw128(X, m, 4 * xb + 3), prmt(c[0].y, c[0].w, 0x7632), prmt(c[1].y, c[1].w, 0x7632),
               prmt(c[2].y, c[2].w, 0x7632), prmt(c[3].y, c[3].w, 0x7632));
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(a_full(a));
        if (gi == 7) mbar_arrive(bar2(3, cs));  // the stage's codes are expanded
      }
    }
  } else {
    // ---- epilogue (warps 0 .. NC / 8 - 1; warp w reads TMEM lanes 32 (w % 4)
    // .. and columns [32 (w / 4), 32 (w / 4 + 1))): accumulator -> registers, the
    // group sums from MMA row 127, the per-group rescale, slice sums folded
    // in slice order in tensor memory, bf16 stores ----
    const int q = warp & 3, hq = warp >> 2;
    const int r = 32 * q + lane;  // TMEM lane = tile row
    const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
    float pacc[CW];
#pragma unroll
    for (int i = 0; i < CW; ++i) pacc[i] = 0.f;
    bool ok = true;
    for (int st = 0; st < ng / 8 && ok; ++st) {
      const int ps = st % PS;
      if (!(ok = wait_all(par_full(ps), (st / PS) & 1))) break;
      const uint32_t prow = params0 + (uint32_t)(ps * kParamTile + r * 16);  // this row's 8 scales, then biases
      // two groups per pass: half the waits, loads and barriers per group
      for (int gi = 0; gi < 8; gi += 2) {
        const int g = 8 * st + gi, b0 = g % NB, b1 = (g + 1) % NB;
        if (!(ok = wait_all(acc_full(b0), (g / NB) & 1) && wait_all(acc_full(b1), ((g + 1) / NB) & 1))) break;
        tc_fence_after_sync();
        float sc[2], cc[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          sc[j] = bf16_bits_to_f32(lds16(prow + 2 * (gi + j)));
          cc[j] = __fmaf_rn(-128.0f, sc[j], bf16_bits_to_f32(lds16(prow + kParamTile / 2 + 2 * (gi + j))));
        }
        const uint32_t sxq0 = sx0 + (uint32_t)((b0 * NC + hq * CW) * 4);
        const uint32_t sxq1 = sx0 + (uint32_t)((b1 * NC + hq * CW) * 4);
#pragma unroll
        for (int c = 0; c < CW; c += 8) {
          float v0[8], v1[8];
          tmem_ld8(tq + (uint32_t)(b0 * NC + hq * CW + c), v0);
          tmem_ld8(tq + (uint32_t)(b1 * NC + hq * CW + c), v1);
          tmem_wait_ld();
          // MMA row 127 (lane 31 of the last lane quarter) holds the group sums
          if (q == 3 && lane == 31) {
            sts128(sxq0 + 4 * c, __float_as_uint(v0[0]), __float_as_uint(v0[1]), __float_as_uint(v0[2]),
                   __float_as_uint(v0[3]));
            sts128(sxq0 + 4 * c + 16, __float_as_uint(v0[4]), __float_as_uint(v0[5]), __float_as_uint(v0[6]),
                   __float_as_uint(v0[7]));
            sts128(sxq1 + 4 * c, __float_as_uint(v1[0]), __float_as_uint(v1[1]), __float_as_uint(v1[2]),
                   __float_as_uint(v1[3]));
            sts128(sxq1 + 4 * c + 16, __float_as_uint(v1[4]), __float_as_uint(v1[5]), __float_as_uint(v1[6]),
                   __float_as_uint(v1[7]));
          }
          named_sync(1 + hq, 128);
#pragma unroll
          for (int i = 0; i < 8; i += 4) {
            const float4 s0 = lds128f(sxq0 + 4 * (c + i));
            const float4 s1 = lds128f(sxq1 + 4 * (c + i));
            const float x0[4] = {s0.x, s0.y, s0.z, s0.w}, x1[4] = {s1.x, s1.y, s1.z, s1.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {  // group g, then group g + 1, per column
              float t = __fmaf_rn(cc[0], x0[k], __fmaf_rn(sc[0], v0[i + k], pacc[c + i + k]));
              pacc[c + i + k] = __fmaf_rn(cc[1], x1[k], __fmaf_rn(sc[1], v1[i + k], t));
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(acc_free(b0));
          mbar_arrive(acc_free(b1));
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(par_free(ps));  // the stage's parameters are read
      const int g = 8 * st + 7;
      if ((g + 1) % p.gps == 0 || g + 1 == ng) {
        // slice end: fold this slice's sums into the running sum, in slice order
        const int slice = g / p.gps;
        const bool last = g + 1 == ng;
        const uint32_t tt = tq + (uint32_t)(NB * NC + hq * CW);
        if (slice > 0) {
#pragma unroll
          for (int c = 0; c < CW; c += 8) {
            float t8[8];
            tmem_ld8(tt + c, t8);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i) pacc[c + i] = __fadd_rn(t8[i], pacc[c + i]);
          }
        }
        if (!last) {
#pragma unroll
          for (int c = 0; c < CW; c += 8) {
            float t8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) t8[i] = pacc[c + i];
            tmem_st8(tt + c, t8);
          }
          tmem_wait_st();
#pragma unroll
          for (int i = 0; i < CW; ++i) pacc[i] = 0.f;
        } else if (r < kTileN) {
          const int n = row0 + r;
#pragma unroll
          for (int i = 0; i < CW; ++i) {
            const int m = col0 + hq * CW + i;
            if (m < p.M && n < p.N) p.y[(int64_t)m * p.N + n] = bf16_rne_bits(pacc[i]);
          }
        }
      }
    }
  }

  // ---- teardown: everything in flight lands before the tensor memory and
  // shared memory are released ----
  __syncthreads();
  if (*s_abort) {
    if (warp == W_PROD && lane == 0) {
      for (int g = issued - S > 0 ? issued - S : 0; g < issued; ++g) mbar_wait_parked(raw_full(g % S), (g / S) & 1);
      const int stages = (issued + 7) / 8;
      for (int st = stages - 2 > 0 ? stages - 2 : 0; st < stages; ++st) mbar_wait_parked(bar2(2, st & 1), (st >> 1) & 1);
      for (int st = stages - PS > 0 ? stages - PS : 0; st < stages; ++st) mbar_wait_parked(par_full(st % PS), (st / PS) & 1);
    }
    if (warp == W_MMA && lane == 0 && mma_done > 0) {
      const int g = mma_done - 1;
      mbar_wait_parked(acc_full(g % NB), (g / NB) & 1);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == W_MMA) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, G::kTmemCols);
  }
}

// ---- host side ------------------------------------------------------------------------

std::mutex g_prefill_mu;
bool g_prefill_attr[64][3] = {};

template <int NC>
cudaError_t prefill_launch_t(const LaunchArgs& a, int gps) {
  using G = PGeo<NC>;
  auto* fn = tc_prefill_kernel<NC>;
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(g_prefill_mu);
    bool& done = g_prefill_attr[dev][NC == 32 ? 0 : NC == 64 ? 1 : 2];
    if (!done) {
      if (cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmem)) return e;
      done = true;
    }
  }
  PrefillMaps maps;
  const int64_t N = a.N, K = a.K;
  if (cudaError_t e = encode_map_2d(&maps.codes, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.Wq, K / 8, N, K / 2, 32, kPRows,
                                    CU_TENSOR_MAP_SWIZZLE_128B))
    return e;
  if (cudaError_t e = encode_map_2d(&maps.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x + (int64_t)a.row0 * K, K, a.M,
                                    2 * K, 64, NC, CU_TENSOR_MAP_SWIZZLE_128B))
    return e;
  if (cudaError_t e = encode_map_2d(&maps.scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.S, K / kGroup, N, K / 32, 8,
                                    kPRows, CU_TENSOR_MAP_SWIZZLE_NONE))
    return e;
  if (cudaError_t e = encode_map_2d(&maps.biases, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.B, K / kGroup, N, K / 32, 8,
                                    kPRows, CU_TENSOR_MAP_SWIZZLE_NONE))
    return e;
  PrefillParams p;
  p.y = a.y + (int64_t)a.row0 * a.N;
  p.flags = a.flags;
  p.N = a.N;
  p.K = a.K;
  p.M = a.M;
  p.groups = a.K / kGroup;
  p.gps = gps;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((a.N + kTileN - 1) / kTileN), (unsigned)((a.M + NC - 1) / NC));
  cfg.blockDim = dim3(G::kThreads);
  cfg.dynamicSmemBytes = (size_t)G::kSmem;
  cfg.stream = a.stream;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, fn, maps, p);
}

}  // namespace

// Many activation rows: one launch covers all M rows, NC at a time per CTA
// column.  The slicing (groups per canonical slice) is that of the skinny
// tensor-core kernels for (N, K), so every row's sums are the same ones.
cudaError_t launch_prefill(const LaunchArgs& a, int slice_k) {
  if (a.K % 512 || slice_k % 512 || a.M < 1) return cudaErrorInvalidValue;
  const int gps = slice_k / kGroup;
  if (a.M <= 32) return prefill_launch_t<32>(a, gps);
  if (a.M <= 64) return prefill_launch_t<64>(a, gps);
  return prefill_launch_t<128>(a, gps);
}

}  // namespace w4a16

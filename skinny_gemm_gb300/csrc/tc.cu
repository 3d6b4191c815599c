// tc.cu -- tensor-core W4A16 skinny GEMM for sm_103a (M = 1..8 per launch).
//
// Citations (page titles; sections in quotes):
//   [W2D2] tiny-llm book, "Week 2 Day 2: Keep W4 Packed"
//   [G4MK] "Gemma 4 E4B & E2B -- single-launch Metal megakernels + lossless
//          speculative decoding" (RESMP-DEV model card)
//
// What it computes: y[m,n] = bf16(sum_g ( s[n,g] * sum_{k in g} x[m,k] q[n,k]
//                                        + b[n,g] * sum_{k in g} x[m,k] ))
// -- the affine identity of [W2D2 "Stage 2: SIMD Matvec"] applied per
// 64-group, with the group sums formed on the tensor cores.
//
// Canonical arithmetic (fixed by (N, K) alone, identical for every M):
//   K is cut into `ksplit` slices of `slice_k` codes.  For one output row and
//   one activation row, a slice partial p_s starts at 0 and, for every
//   64-group of the slice in order,
//       acc = sum_{k in group} x_k (128 + q_k)   (four m16n8k16 MMAs, fp32)
//       sx  = sum_{k in group} x_k               (four MMAs with A = 1.0)
//       p_s = fma(s, acc, p_s);  p_s = fma(b - 128 s, sx, p_s)
//   and y = bf16(((p_0 + p_1) + p_2) + ...).  Every kernel in this file
//   reproduces exactly this sequence, so row m of any call equals the M = 1
//   call bit for bit ([G4MK "Implementation notes": the verify GEMM is kept
//   arithmetic-identical to the sequential GEMV), and w4a16_mm_id rows equal
//   w4a16_mm on the selected expert.  An MMA output column depends only on
//   its own activation column, so unused columns (M < 8) change nothing.
//
// Data path of one warp:
//  * Packed codes stream HBM -> shared memory by TMA (cp.async.bulk.tensor,
//    128-byte swizzle), 32 rows x 256 codes (4 KB) per stage, into a ring of
//    `stages` slots, each guarded by an mbarrier.  The stage's activation
//    chunk (M rows x 256 bf16) arrives by cp.async.bulk into padded rows of
//    the same slot.  Lane 0 issues both; the ring runs ahead across work
//    units, so DRAM latency is paid once per warp, not once per tile.
//  * ldmatrix.x4 hands every lane, for rows g and g+8 of a 16-row subtile,
//    the packed words the m16n8k16 A fragment needs (bank-conflict free
//    thanks to the swizzle).
//  * One LOP3 per pair of codes ORs two nibbles into the mantissas of bf16
//    128.0 (0x4300): exact 128+q, no subtraction; the 128 offset is folded
//    into the group bias above (b - 128 s is exact in fp32 for bf16 s, b).
//  * The order of K inside an MMA is a fixed permutation (each lane pairs
//    codes i and i+4 of a packed word); the activations are permuted the
//    same way with PRMT, so each dot product is unchanged.
//
// w4a16_mm runs a persistent grid: work units (32 rows x one K-slice) are
// dealt round-robin to warps, which gives every SM the same share of bytes
// whatever N is.  With ksplit > 1 a unit writes its fp32 partial to a
// workspace and bumps a per-tile counter; the warp that completes a tile
// adds the partials in slice order (the result does not depend on which
// warp arrives last) and resets the counter.  w4a16_mm_id runs one CTA per
// (row tile, expert); its warps compute whole slices and add them in slice
// order in shared memory.
//
// No spin-wait is unbounded: an mbarrier wait that exceeds its iteration
// limit raises W4A16_DEVICE_TIMEOUT and the warp stops computing.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "launch.h"
#include "route.cuh"

namespace w4a16 {
namespace {

constexpr int kTileRows = 32;           // two m16 subtiles per warp
constexpr int kStageK = 256;            // codes per stage per row (one 128-byte box row)
constexpr int kStageWords = kStageK / 8;
constexpr int kCodeSlotBytes = kTileRows * kStageWords * 4;  // 4096
constexpr int kXPitch = kStageK * 2 + 64;                     // 576: conflict-free LDS.128
constexpr int kStreamWarps = 4;          // warps per CTA of the persistent kernel
constexpr int kRoutedWarps = 8;          // max warps per CTA of the routed kernel
constexpr int kTargetUnits = 152 * 16;   // work units wanted per chunk (~16 per SM)
constexpr int kSmemLimit = 227 * 1024;
constexpr uint32_t kWaitLimit = 1u << 20;
constexpr uint32_t kMagic = 0x43004300u;  // two bf16 128.0
constexpr uint32_t kOnes = 0x3F803F80u;   // two bf16 1.0

// ---- PTX wrappers -------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: true when the phase completed, false after kWaitLimit tries.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Pass a shared-memory address through an ordered instruction, so loads that
// use the result cannot be scheduled before the preceding barrier wait.
__device__ __forceinline__ uint32_t ordered(uint32_t v) {
  uint32_t r;
  asm volatile("mov.b32 %0, %1;" : "=r"(r) : "r"(v) : "memory");
  return r;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int cx, int cy, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(map), "r"(cx), "r"(cy), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// (w & 0x000F000F) | 0x43004300 : nibbles 0 and 4 of w as bf16 128+q.
__device__ __forceinline__ uint32_t codes_as_bf16x2(uint32_t w) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(w), "r"(0x000F000Fu), "r"(kMagic));
  return d;
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint2 ldg_params(const uint16_t* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ float half_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float half_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// ---- one warp's stage ring -------------------------------------------------------------

struct Ring {
  uint32_t codes0, xs0, bars0;
  int S, x_slot;
  uint32_t issued, consumed;
};

// Lane 0 only: start the loads of one stage (codes of rows tensor_row.., x of
// the listed activation rows) into the next free slot.
__device__ __forceinline__ void ring_issue(Ring& R, const CUtensorMap* map, int st, int tensor_row,
                                           const uint16_t* x, const int* toks, int mc, int K) {
  const uint32_t slot = R.issued % (uint32_t)R.S;
  const uint32_t bar = R.bars0 + 8 * slot;
  mbar_expect_tx(bar, kCodeSlotBytes + (uint32_t)(mc * kStageK * 2));
  tma_load_2d(R.codes0 + slot * kCodeSlotBytes, map, st * kStageWords, tensor_row, bar);
  for (int n = 0; n < mc; ++n)
    bulk_load(R.xs0 + slot * R.x_slot + n * kXPitch, x + (int64_t)toks[n] * K + (int64_t)st * kStageK,
              kStageK * 2, bar);
  ++R.issued;
}

// All lanes: wait for the oldest outstanding slot.  Returns false on timeout.
__device__ __forceinline__ bool ring_wait(Ring& R, uint32_t& slot) {
  slot = R.consumed % (uint32_t)R.S;
  const uint32_t parity = (R.consumed / (uint32_t)R.S) & 1u;
  const bool ok = mbar_wait(R.bars0 + 8 * slot, parity);
  return __all_sync(0xffffffffu, ok);
}

// Group parameters (scale, bias) of the 4 groups of stage `st` for this
// lane's rows prow[i] (matrix rows; rows >= N read nothing).
__device__ __forceinline__ void load_params(const uint16_t* Se, const uint16_t* Be, const int (&prow)[4], int N,
                                            int groups_per_row, int st, uint2 (&sv)[4], uint2 (&bv)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (prow[i] < N) {
      const int64_t off = (int64_t)prow[i] * groups_per_row + st * (kStageK / kGroup);
      sv[i] = ldg_params(Se + off);
      bv[i] = ldg_params(Be + off);
    } else {
      sv[i] = make_uint2(0, 0);
      bv[i] = make_uint2(0, 0);
    }
  }
}

// One stage (32 rows x 256 codes) of the canonical recurrence into p[s][i]:
// subtile s, i = (row g: tokens 2t, 2t+1; row g+8: tokens 2t, 2t+1).
__device__ __forceinline__ void compute_stage(uint32_t cbase, uint32_t xbase, bool xvalid, const uint2 (&ps)[4],
                                              const uint2 (&pb)[4], float (&p)[2][4], int lane) {
#pragma unroll
  for (int gi = 0; gi < 4; ++gi) {
    uint32_t bx[2][2][2];
#pragma unroll
    for (int cb = 0; cb < 2; ++cb) {
      uint4 u = make_uint4(0, 0, 0, 0);
      if (xvalid) u = lds128(xbase + 128 * gi + 64 * cb);
      bx[cb][0][0] = prmt(u.x, u.z, 0x5410);
      bx[cb][0][1] = prmt(u.x, u.z, 0x7632);
      bx[cb][1][0] = prmt(u.y, u.w, 0x5410);
      bx[cb][1][1] = prmt(u.y, u.w, 0x7632);
    }
    float sx[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int cb = 0; cb < 2; ++cb)
#pragma unroll
      for (int h = 0; h < 2; ++h) mma_bf16(sx, kOnes, kOnes, kOnes, kOnes, bx[cb][h][0], bx[cb][h][1]);

#pragma unroll
    for (int s = 0; s < 2; ++s) {
      uint32_t w[4];  // rows g / g+8 for chunk 2gi, then for chunk 2gi+1
      {
        const int mi = lane >> 3, r8 = lane & 7;
        const int row = 16 * s + 8 * (mi & 1) + r8;
        const int chunk = 2 * gi + (mi >> 1);
        ldsm_x4(cbase + row * 128 + ((chunk ^ (row & 7)) << 4), w[0], w[1], w[2], w[3]);
      }
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int cb = 0; cb < 2; ++cb) {
        const uint32_t wg = w[2 * cb], wg8 = w[2 * cb + 1];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t a0 = codes_as_bf16x2(wg >> (8 * h));
          const uint32_t a1 = codes_as_bf16x2(wg8 >> (8 * h));
          const uint32_t a2 = codes_as_bf16x2(wg >> (8 * h + 4));
          const uint32_t a3 = codes_as_bf16x2(wg8 >> (8 * h + 4));
          mma_bf16(acc, a0, a1, a2, a3, bx[cb][h][0], bx[cb][h][1]);
        }
      }
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int i = 2 * s + rr;
        const uint32_t sw = (gi < 2) ? ps[i].x : ps[i].y;
        const uint32_t bw = (gi < 2) ? pb[i].x : pb[i].y;
        const float sc = (gi & 1) ? half_hi(sw) : half_lo(sw);
        const float bi = (gi & 1) ? half_hi(bw) : half_lo(bw);
        const float cc = __fmaf_rn(-128.0f, sc, bi);
        p[s][2 * rr + 0] = __fmaf_rn(sc, acc[2 * rr + 0], p[s][2 * rr + 0]);
        p[s][2 * rr + 0] = __fmaf_rn(cc, sx[0], p[s][2 * rr + 0]);
        p[s][2 * rr + 1] = __fmaf_rn(sc, acc[2 * rr + 1], p[s][2 * rr + 1]);
        p[s][2 * rr + 1] = __fmaf_rn(cc, sx[1], p[s][2 * rr + 1]);
      }
    }
  }
}

struct Shape {
  int nst, tiles, sl, ks, units;
};

__host__ __device__ inline Shape tc_shape(int N, int K) {
  Shape s;
  s.nst = K / kStageK;
  s.tiles = (N + kTileRows - 1) / kTileRows;
  int64_t sl = (int64_t)s.nst * s.tiles / kTargetUnits;
  if (sl < 1) sl = 1;
  if (sl > s.nst) sl = s.nst;
  s.sl = (int)sl;
  s.ks = (s.nst + s.sl - 1) / s.sl;
  s.units = s.tiles * s.ks;
  return s;
}

__host__ __device__ inline int ring_bytes(int stages, int mcap) {
  return stages * (kCodeSlotBytes + mcap * kXPitch);
}

// ---- persistent kernel (w4a16_mm) ------------------------------------------------------

struct StreamParams {
  const uint16_t* x;
  const uint16_t* S;
  const uint16_t* B;
  uint16_t* y;
  float* part;      // [units][8][32] slice partials (ksplit > 1)
  int* cnt;         // [tiles] arrival counters, zero between launches
  int* flags;
  int N, K, M, row0;
  int nst, sl, ks, tiles, units;
  int stages;
};

__global__ void __launch_bounds__(kStreamWarps * 32, 3) tc_stream_kernel(const __grid_constant__ CUtensorMap tmW,
                                                                      StreamParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int S = p.stages, mc = p.M;
  const int x_slot = mc * kXPitch;
  const int groups_per_row = p.K / kGroup;

  // layout: codes ring of every warp | x ring of every warp | barriers | tokens
  Ring R;
  R.S = S;
  R.x_slot = x_slot;
  R.codes0 = smem_u32(base) + (uint32_t)(warp * S * kCodeSlotBytes);
  R.xs0 = smem_u32(base) + (uint32_t)(kStreamWarps * S * kCodeSlotBytes + warp * S * x_slot);
  const uint32_t bar_off = (uint32_t)(kStreamWarps * ring_bytes(S, mc));
  R.bars0 = smem_u32(base) + bar_off + (uint32_t)(warp * S * 8);
  int* s_tok = reinterpret_cast<int*>(base + bar_off + kStreamWarps * S * 8);
  R.issued = R.consumed = 0;

  if (lane == 0)
    for (int i = 0; i < S; ++i) mbar_init(R.bars0 + 8 * i, 1);
  if (threadIdx.x < mc) s_tok[threadIdx.x] = p.row0 + threadIdx.x;
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();

  // warp-major numbering: every pass over the units spreads them evenly over CTAs
  const int gw = warp * gridDim.x + blockIdx.x;
  const int TW = gridDim.x * kStreamWarps;
  if (gw >= p.units) return;

  // issue cursor: unit iu, stage ist (stages of a unit are [slice*sl, ...))
  int iu = gw;
  int ist = (iu % p.ks) * p.sl;
  auto unit_end = [&](int u) {
    const int e = (u % p.ks + 1) * p.sl;
    return e < p.nst ? e : p.nst;
  };
  auto issue_next = [&]() {
    if (iu >= p.units) return;
    ring_issue(R, &tmW, ist, (iu / p.ks) * kTileRows, p.x, s_tok, mc, p.K);
    if (++ist == unit_end(iu)) {
      iu += TW;
      if (iu < p.units) ist = (iu % p.ks) * p.sl;
    }
  };
  if (lane == 0) {
    fence_proxy_async();
    for (int i = 0; i < S; ++i) issue_next();
  }

  bool timed_out = false;
  int pend_tile = -1, pend_old = 0;

  auto reduce_tile = [&](int tile) {
    // Sum the ksplit partials of a finished tile in slice order.
    __threadfence();
    const int row = tile * kTileRows + lane;
    for (int n = 0; n < mc; ++n) {
      const float* q = p.part + ((int64_t)tile * p.ks * 8 + n) * 32 + lane;
      float sum = __ldcg(q);
      for (int sidx = 1; sidx < p.ks; ++sidx) sum = __fadd_rn(sum, __ldcg(q + (int64_t)sidx * 8 * 32));
      if (row < p.N) p.y[(int64_t)s_tok[n] * p.N + row] = f32_to_bf16_bits(sum);
    }
    if (lane == 0) p.cnt[tile] = 0;
  };

  for (int u = gw; u < p.units && !timed_out; u += TW) {
    const int tile = u / p.ks, slice = u % p.ks;
    const int s0 = slice * p.sl, s1 = unit_end(u);
    int prow[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) prow[i] = tile * kTileRows + 16 * (i >> 1) + g + 8 * (i & 1);

    float acc[2][4];
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[s][i] = 0.0f;

    uint2 ps[4], pb[4];
    load_params(p.S, p.B, prow, p.N, groups_per_row, s0, ps, pb);
    for (int st = s0; st < s1; ++st) {
      uint32_t slot;
      if (!ring_wait(R, slot)) {
        timed_out = true;
        break;
      }
      uint2 ns[4] = {}, nb[4] = {};
      if (st + 1 < s1) load_params(p.S, p.B, prow, p.N, groups_per_row, st + 1, ns, nb);
      const uint32_t cbase = ordered(R.codes0 + slot * kCodeSlotBytes);
      const uint32_t xbase = ordered(R.xs0 + slot * x_slot + g * kXPitch + 16 * t);
      compute_stage(cbase, xbase, g < mc, ps, pb, acc, lane);
      ++R.consumed;
      __syncwarp();
      if (lane == 0) {
        fence_proxy_async();
        issue_next();
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        ps[i] = ns[i];
        pb[i] = nb[i];
      }
    }
    if (timed_out) break;

    // the previous unit's arrival count has had a whole unit to come back
    if (pend_tile >= 0) {
      const int old = __shfl_sync(0xffffffffu, pend_old, 0);
      if (old == p.ks - 1) reduce_tile(pend_tile);
      pend_tile = -1;
    }
    if (p.ks == 1) {
#pragma unroll
      for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = prow[2 * s + (i >> 1)];
          const int n = 2 * t + (i & 1);
          if (n < mc && row < p.N) p.y[(int64_t)s_tok[n] * p.N + row] = f32_to_bf16_bits(acc[s][i]);
        }
    } else {
      float* q = p.part + (int64_t)u * 8 * 32;
#pragma unroll
      for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 16 * s + g + 8 * (i >> 1);
          const int n = 2 * t + (i & 1);
          if (n < mc) __stcg(q + n * 32 + r, acc[s][i]);
        }
      __threadfence();
      __syncwarp();
      if (lane == 0) pend_old = atomicAdd(p.cnt + tile, 1);
      pend_tile = tile;
    }
  }
  if (!timed_out && pend_tile >= 0) {
    const int old = __shfl_sync(0xffffffffu, pend_old, 0);
    if (old == p.ks - 1) reduce_tile(pend_tile);
  }
  if (timed_out) {
    if (lane == 0) atomicOr(p.flags, W4A16_DEVICE_TIMEOUT);
    // let copies already in flight land before shared memory is released
    while (R.consumed < R.issued) {
      mbar_wait(R.bars0 + 8 * (R.consumed % (uint32_t)S), (R.consumed / (uint32_t)S) & 1u);
      ++R.consumed;
    }
  }
}

// ---- routed kernel (w4a16_mm_id) -------------------------------------------------------

struct RoutedParams {
  const uint16_t* x;
  const uint16_t* S;
  const uint16_t* B;
  uint16_t* y;
  const int32_t* ids;
  int* flags;
  int N, K, T, E;
  int nst, sl, ks;
  int warps, stages;
};

__host__ __device__ inline int routed_smem(int warps, int stages, int ks) {
  return warps * ring_bytes(stages, kMaxChunk) + warps * stages * 8 + ks * kTileRows * 8 * 4 + 16 * 4 + 1024;
}

__global__ void __launch_bounds__(kRoutedWarps * 32) tc_routed_kernel(const __grid_constant__ CUtensorMap tmW,
                                                                      RoutedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int S = p.stages, W = p.warps;
  const int x_slot = kMaxChunk * kXPitch;
  const int groups_per_row = p.K / kGroup;
  const int e = blockIdx.y;
  const int row_base = blockIdx.x * kTileRows;
  const int tensor_row = e * p.N + row_base;
  const uint16_t* Se = p.S + (int64_t)e * p.N * groups_per_row;
  const uint16_t* Be = p.B + (int64_t)e * p.N * groups_per_row;

  Ring R;
  R.S = S;
  R.x_slot = x_slot;
  R.codes0 = smem_u32(base) + (uint32_t)(warp * S * kCodeSlotBytes);
  R.xs0 = smem_u32(base) + (uint32_t)(W * S * kCodeSlotBytes + warp * S * x_slot);
  const uint32_t bar_off = (uint32_t)(W * ring_bytes(S, kMaxChunk));
  R.bars0 = smem_u32(base) + bar_off + (uint32_t)(warp * S * 8);
  float* red = reinterpret_cast<float*>(base + bar_off + W * S * 8);  // [ks][32 rows][8 tokens]
  int* s_tok = reinterpret_cast<int*>(red + p.ks * kTileRows * 8);
  int* s_state = s_tok + kMaxChunk;  // [0] scan position, [1] count, [2] abort
  R.issued = R.consumed = 0;

  if (lane == 0)
    for (int i = 0; i < S; ++i) mbar_init(R.bars0 + 8 * i, 1);
  if (threadIdx.x == 0) {
    s_state[0] = 0;
    s_state[2] = 0;
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();

  int prow[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) prow[i] = row_base + 16 * (i >> 1) + g + 8 * (i & 1);

  // this warp's stages: slices warp, warp + W, ... each [slice*sl, min(nst, ...))
  auto slice_end = [&](int sidx) {
    const int e2 = (sidx + 1) * p.sl;
    return e2 < p.nst ? e2 : p.nst;
  };

  for (;;) {
    const int mc = gather_tokens(p.ids, p.T, p.E, e, s_tok, s_state);
    if (mc == 0) break;

    int isl = warp, ist = warp * p.sl;  // issue cursor
    auto issue_next = [&]() {
      if (isl >= p.ks) return;
      ring_issue(R, &tmW, ist, tensor_row, p.x, s_tok, mc, p.K);
      if (++ist == slice_end(isl)) {
        isl += W;
        ist = isl * p.sl;
      }
    };
    if (lane == 0) {
      fence_proxy_async();
      for (int i = 0; i < S; ++i) issue_next();
    }
    bool timed_out = false;
    for (int sidx = warp; sidx < p.ks && !timed_out; sidx += W) {
      float acc[2][4];
#pragma unroll
      for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[s][i] = 0.0f;
      const int s0 = sidx * p.sl, s1 = slice_end(sidx);
      uint2 ps[4], pb[4];
      load_params(Se, Be, prow, p.N, groups_per_row, s0, ps, pb);
      for (int st = s0; st < s1; ++st) {
        uint32_t slot;
        if (!ring_wait(R, slot)) {
          timed_out = true;
          break;
        }
        uint2 ns[4] = {}, nb[4] = {};
        if (st + 1 < s1) load_params(Se, Be, prow, p.N, groups_per_row, st + 1, ns, nb);
        const uint32_t cbase = ordered(R.codes0 + slot * kCodeSlotBytes);
        const uint32_t xbase = ordered(R.xs0 + slot * x_slot + g * kXPitch + 16 * t);
        compute_stage(cbase, xbase, g < mc, ps, pb, acc, lane);
        ++R.consumed;
        __syncwarp();
        if (lane == 0) {
          fence_proxy_async();
          issue_next();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ps[i] = ns[i];
          pb[i] = nb[i];
        }
      }
      float* rs = red + sidx * kTileRows * 8;
#pragma unroll
      for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int i = 0; i < 4; ++i) rs[(16 * s + g + 8 * (i >> 1)) * 8 + 2 * t + (i & 1)] = acc[s][i];
    }
    if (timed_out) {
      if (lane == 0) {
        atomicOr(p.flags, W4A16_DEVICE_TIMEOUT);
        s_state[2] = 1;
      }
      while (R.consumed < R.issued) {
        mbar_wait(R.bars0 + 8 * (R.consumed % (uint32_t)S), (R.consumed / (uint32_t)S) & 1u);
        ++R.consumed;
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kTileRows * 8; i += blockDim.x) {
      const int r = i >> 3, n = i & 7;
      const int row = row_base + r;
      if (n < mc && row < p.N) {
        float sum = red[r * 8 + n];
        for (int sidx = 1; sidx < p.ks; ++sidx) sum = __fadd_rn(sum, red[(sidx * kTileRows + r) * 8 + n]);
        p.y[(int64_t)s_tok[n] * p.N + row] = f32_to_bf16_bits(sum);
      }
    }
    __syncthreads();
    if (s_state[2]) break;  // CTA-uniform
  }

  if (e == 0 && !s_state[2]) {
    // tokens whose expert id is out of range: zero rows, raise the flag
    if (threadIdx.x == 0) s_state[0] = 0;
    __syncthreads();
    for (;;) {
      const int cnt = gather_tokens(p.ids, p.T, p.E, -1, s_tok, s_state);
      if (cnt == 0) break;
      if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(p.flags, W4A16_DEVICE_BAD_ID);
      for (int i = threadIdx.x; i < cnt * kTileRows; i += blockDim.x) {
        const int row = row_base + i % kTileRows;
        if (row < p.N) p.y[(int64_t)s_tok[i / kTileRows] * p.N + row] = 0;
      }
      __syncthreads();
    }
  }
}

// ---- host side ------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_status = cudaSuccess;

cudaError_t get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
      g_encode_status = (e != cudaSuccess) ? e : cudaErrorNotSupported;
      return;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode_status;
}

cudaError_t make_code_map(CUtensorMap* map, const uint32_t* Wq, int64_t rows, int K) {
  if (cudaError_t e = get_encoder()) return e;
  cuuint64_t dims[2] = {(cuuint64_t)(K / 8), (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K / 2};
  cuuint32_t box[2] = {(cuuint32_t)kStageWords, (cuuint32_t)kTileRows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(Wq), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int stream_smem(int stages, int mc) {
  return kStreamWarps * ring_bytes(stages, mc) + kStreamWarps * stages * 8 + 64 + 1024;
}

// Deepest ring (4..2 stages per warp) that still lets three CTAs share an SM.
int stream_stages(int mc) {
  for (int s = 4; s > 2; --s)
    if (stream_smem(s, mc) <= 76 * 1024) return s;
  return 2;
}

struct DeviceInfo {
  int sms = 152;
  bool attr_set[2] = {false, false};
};

std::mutex g_dev_mu;
std::map<int, DeviceInfo> g_dev;

DeviceInfo& device_info(int dev) {
  auto it = g_dev.find(dev);
  if (it == g_dev.end()) {
    DeviceInfo d;
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) d.sms = v;
    it = g_dev.emplace(dev, d).first;
  }
  return it->second;
}

// Workspace of one (device, stream), fixed layout:
//   [kWsTiles] int arrival counters (zero between launches) | [kWsUnits][8][32] fp32 slice partials.
// ksplit > 1 only happens when a chunk has fewer than kTargetUnits row tiles,
// and then it never has more than kWsUnits work units (checked at launch), so
// one fixed-size buffer serves every shape and never needs to grow.
constexpr int kWsTiles = 4096;
constexpr int kWsUnits = 4864;
constexpr size_t kWsCounterBytes = (size_t)kWsTiles * 4;
constexpr size_t kWsBytes = kWsCounterBytes + (size_t)kWsUnits * 8 * 32 * 4;

struct Workspace {
  void* ptr = nullptr;
};
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

cudaError_t workspace(int dev, cudaStream_t stream, void** out) {
  Workspace& w = g_ws[{dev, stream}];
  if (w.ptr) {
    *out = w.ptr;
    return cudaSuccess;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone)
    return cudaErrorStreamCaptureUnsupported;  // allocate only outside capture
  void* p = nullptr;
  if (cudaError_t e = cudaMalloc(&p, kWsBytes)) return e;
  if (cudaError_t e = cudaMemsetAsync(p, 0, kWsCounterBytes, stream)) {
    cudaFree(p);
    return e;
  }
  w.ptr = p;
  *out = p;
  return cudaSuccess;
}

}  // namespace

bool tc_supported(int N, int K) {
  (void)N;
  return K % kStageK == 0;
}

void plan_tc(int N, int K, w4a16_plan* p) {
  const Shape s = tc_shape(N, K);
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    sms = device_info(dev).sms;
  } else {
    cudaGetLastError();
  }
  const int smem = stream_smem(stream_stages(1), 1);
  const int per_sm = kSmemLimit / smem > 0 ? kSmemLimit / smem : 1;
  int grid = sms * per_sm;
  const int need = (s.units + kStreamWarps - 1) / kStreamWarps;
  if (grid > need) grid = need;
  p->kernel = W4A16_KERNEL_TC;
  p->ksplit = s.ks;
  p->slice_k = s.sl * kStageK;
  p->rows_per_tile = kTileRows;
  p->units = s.units;
  p->threads = kStreamWarps * 32;
  p->grid_x = grid;
  p->smem_bytes = smem;
}

cudaError_t launch_tc(const LaunchArgs& a, const w4a16_plan& plan) {
  (void)plan;
  const Shape s = tc_shape(a.N, a.K);
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  StreamParams p;
  p.x = a.x; p.S = a.S; p.B = a.B; p.y = a.y; p.flags = a.flags;
  p.N = a.N; p.K = a.K; p.M = a.M; p.row0 = a.row0;
  p.nst = s.nst; p.sl = s.sl; p.ks = s.ks; p.tiles = s.tiles; p.units = s.units;
  p.stages = stream_stages(a.M);
  p.part = nullptr;
  p.cnt = nullptr;
  int sms;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = device_info(dev);
    sms = d.sms;
    if (!d.attr_set[0]) {
      if (cudaError_t e = cudaFuncSetAttribute(tc_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kSmemLimit))
        return e;
      d.attr_set[0] = true;
    }
    if (s.ks > 1) {
      if (s.tiles > kWsTiles || s.units > kWsUnits) return cudaErrorInvalidValue;
      void* ws = nullptr;
      if (cudaError_t e = workspace(dev, a.stream, &ws)) return e;
      p.cnt = static_cast<int*>(ws);
      p.part = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsCounterBytes);
    }
  }
  CUtensorMap map;
  if (cudaError_t e = make_code_map(&map, a.Wq, a.N, a.K)) return e;
  const int smem = stream_smem(p.stages, a.M);
  int per_sm = 0;
  if (cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc_stream_kernel, kStreamWarps * 32, smem))
    return e;
  if (per_sm < 1) per_sm = 1;
  int grid = sms * per_sm;
  const int need = (s.units + kStreamWarps - 1) / kStreamWarps;
  if (grid > need) grid = need;
  tc_stream_kernel<<<grid, kStreamWarps * 32, smem, a.stream>>>(map, p);
  return cudaGetLastError();
}

cudaError_t launch_tc_id(const LaunchArgs& a, const w4a16_plan& plan) {
  (void)plan;
  const Shape s = tc_shape(a.N, a.K);
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  RoutedParams p;
  p.x = a.x; p.S = a.S; p.B = a.B; p.y = a.y; p.ids = a.ids; p.flags = a.flags;
  p.N = a.N; p.K = a.K; p.T = a.T; p.E = a.E;
  p.nst = s.nst; p.sl = s.sl; p.ks = s.ks;
  p.warps = s.ks < kRoutedWarps ? s.ks : kRoutedWarps;
  p.stages = 3;
  while (p.stages > 2 && routed_smem(p.warps, p.stages, p.ks) > kSmemLimit) --p.stages;
  while (p.warps > 1 && routed_smem(p.warps, p.stages, p.ks) > kSmemLimit) --p.warps;
  const int smem = routed_smem(p.warps, p.stages, p.ks);
  if (smem > kSmemLimit) return cudaErrorInvalidConfiguration;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = device_info(dev);
    if (!d.attr_set[1]) {
      if (cudaError_t e = cudaFuncSetAttribute(tc_routed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kSmemLimit))
        return e;
      d.attr_set[1] = true;
    }
  }
  CUtensorMap map;
  if (cudaError_t e = make_code_map(&map, a.Wq, (int64_t)a.N * a.E, a.K)) return e;
  dim3 grid(s.tiles, a.E);
  tc_routed_kernel<<<grid, p.warps * 32, smem, a.stream>>>(map, p);
  return cudaGetLastError();
}


// ---- no-allocation variant ----------------------------------------------------------------
//
// Some callers may not call cudaMalloc at all: code that runs inside an
// engine which reserved all device memory up front and hands out nothing
// else, processes under a hard device-memory cap where a late allocation can
// fail in the middle of serving, and deployments that forbid any allocation
// after start-up.  For them w4a16_mm_noalloc runs the same persistent kernel
// as w4a16_mm, but its split-K workspace is this fixed array, which every GPU
// that loads the library holds until the process exits.
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[kWsBytes];

// Device address of g_noalloc_scratch, looked up once per device.  In host
// code the array's name is only a stand-in for the symbol, never a pointer a
// kernel may use.
void* g_noalloc_ptr[64] = {};

}  // namespace

size_t tc_noalloc_scratch_bytes() { return kWsBytes; }

bool tc_noalloc_fits(int N, int K) {
  const Shape s = tc_shape(N, K);
  return s.ks == 1 || (s.tiles <= kWsTiles && s.units <= kWsUnits);
}

cudaError_t launch_tc_noalloc(const LaunchArgs& a) {
  const Shape s = tc_shape(a.N, a.K);
  if (s.ks > 1 && (s.tiles > kWsTiles || s.units > kWsUnits)) return cudaErrorInvalidValue;
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int sms;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = device_info(dev);
    sms = d.sms;
    if (!d.attr_set[0]) {
      if (cudaError_t e = cudaFuncSetAttribute(tc_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kSmemLimit))
        return e;
      d.attr_set[0] = true;
    }
    if (!g_noalloc_ptr[dev]) {
      void* ptr = nullptr;
      if (cudaError_t e = cudaGetSymbolAddress((void**)&ptr, g_noalloc_scratch)) return e;
      g_noalloc_ptr[dev] = ptr;
    }
    scratch = g_noalloc_ptr[dev];
  }
  StreamParams p;
  p.x = a.x; p.S = a.S; p.B = a.B; p.y = a.y; p.flags = a.flags;
  p.N = a.N; p.K = a.K; p.M = a.M; p.row0 = a.row0;
  p.nst = s.nst; p.sl = s.sl; p.ks = s.ks; p.tiles = s.tiles; p.units = s.units;
  p.stages = stream_stages(a.M);
  p.part = nullptr;
  p.cnt = nullptr;
  if (s.ks > 1) {
    p.cnt = static_cast<int*>(scratch);
    p.part = reinterpret_cast<float*>(static_cast<char*>(scratch) + kWsCounterBytes);
    // the array keeps whatever the previous call left: the counters must start at zero
    if (cudaError_t e = cudaMemsetAsync(p.cnt, 0, (size_t)s.tiles * 4, a.stream)) return e;
  }
  CUtensorMap map;
  if (cudaError_t e = make_code_map(&map, a.Wq, a.N, a.K)) return e;
  const int smem = stream_smem(p.stages, a.M);
  int per_sm = 0;
  if (cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc_stream_kernel, kStreamWarps * 32, smem))
    return e;
  if (per_sm < 1) per_sm = 1;
  int grid = sms * per_sm;
  const int need = (s.units + kStreamWarps - 1) / kStreamWarps;
  if (grid > need) grid = need;
  tc_stream_kernel<<<grid, kStreamWarps * 32, smem, a.stream>>>(map, p);
  return cudaGetLastError();
}

}  // namespace w4a16

// stq1.cu -- the STQ1_0 ternary matmul (sm_103a).
//
// "Hy4-preview Metal kernels for llama.cpp" gives the format (section "Notes
// and gotchas": 42-byte blocks of 256 weights, 4-bit group codes, group sign
// bits, an fp16 scale, and the weight-to-group map), the kernels a model
// needs (the kernel table: matvec, small batches, routed experts, row
// gather) and the structure of a group (section "Results", the fourth decode
// pass: one zero lane named by the code's high bits, two sign flips in its
// low bits, the sign bit negating the group).  Its results also found a
// table lookup faster than decoding the weights arithmetically.  Here the
// table sits on the activation side:
//
//  * The four weights of a group take one of 32 patterns (16 codes, each
//    with or without the group sign), so the group's share of an output is
//    one of 32 signed sums of its four activations.  A CTA writes those sums
//    for the groups of a stretch of K into shared memory, once per
//    activation row; each weight row then adds, per group, the entry its code
//    and sign bit select.  Per group and weight row that is a byte extract,
//    an address multiply-add, and per activation row one shared load and one
//    add.  Entries with the sign set are exact negations.
//  * A lane owns one weight row: 32 rows per warp, 256 per CTA, so every
//    entry serves 256 rows.  The weights stream as records of 16 rows x one
//    block (the page's bytes regrouped by stq1_pack so that a row's codes,
//    sign bits and scale are contiguous) through a ring of bulk copies
//    (cp.async.bulk on an mbarrier) per warp.
//  * K is split over a cluster of up to 8 CTAs (a function of (N, K)); the
//    slice sums meet in the first CTA's shared memory and are added there in
//    slice order.
//
// Arithmetic, every order fixed by (N, K) (so any row of a multi-row call
// equals the one-row call, and routed rows equal stq1_mm on their expert):
//   entry of code c, nonzero lanes p < q < r:  (x_r + e_q x_q) + e_p x_p
//   block sum:  (s_0 + s_1) + (s_2 + s_3), s_i = the groups g = i (mod 4) in order
//   slice sum:  t = fma(d_b, block sum_b, t) over the slice's blocks in order
//   output:     ((t_0 + t_1) + t_2) + ... over the slices
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "ptx.cuh"
#include "stq1.cuh"
#include "w4a16.h"

namespace w4a16 {
namespace {

using namespace ptx;

constexpr int kBlockW = 256;     // weights per block
constexpr int kBlockBytes = 42;  // bytes per block in the page's layout
// One record: 16 rows x one block, 672 bytes.  Codes [2 halves][16 rows][16]
// (qs bytes 16h .. 16h + 15 of row r at 256 h + 16 r), sign bytes [16 rows][8]
// at 512, scales [16 rows][2] at 640.
constexpr int kRec = 672;
constexpr int kSignOff = 512;
constexpr int kScaleOff = 640;
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kRowsCta = 32 * kWarps;  // one weight row per lane
constexpr int kDepth = 4;              // blocks in flight per warp
constexpr int kSlot = 2 * kRec;        // one block of a warp's two 16-row tiles
constexpr int kMaxRows = 8;            // activation rows per pass
constexpr int kMaxCluster = 8;
constexpr int kMaxSpc = 4;  // K slices one CTA may take
constexpr int kWaveCtas = 256;         // CTAs that surely run at once (two per SM, clusters packed)

// Table of one pass of MR activation rows over (8 / MR) blocks: per row and
// block kTabBlock bytes (33 x 256, so every block starts 256-byte aligned);
// in a block the 32 pairs of groups (2q, 2q + 1) are kPairBytes apart, the
// even group's 32 entries (one per label) at 0, the odd group's at 128.  A
// lookup address is then the block's base with its low byte replaced by the
// label's byte offset (one byte permute) plus an immediate; the pair stride
// (65 words) puts the 32 labels of a group in 32 distinct banks.  The table
// area starts at the first 256-byte boundary of the dynamic shared memory.
constexpr int kPairBytes = 260;
constexpr int kTabBlock = 33 * 256;
__host__ __device__ constexpr int tab_blocks(int mr) { return 8 / mr; }
__host__ __device__ constexpr int tab_row_bytes(int mr) { return tab_blocks(mr) * kTabBlock; }
__host__ __device__ constexpr int tab_bytes(int mr) { return mr * tab_row_bytes(mr) + 256; }
__host__ __device__ constexpr int ring_off(int mr) { return (tab_bytes(mr) + 127) & ~127; }
__host__ __device__ constexpr int bar_off(int mr) { return ring_off(mr) + kWarps * kDepth * kSlot; }
__host__ __device__ constexpr int tok_off(int mr) { return bar_off(mr) + kWarps * kDepth * 8; }
__host__ __device__ constexpr int smem_bytes(int mr) { return tok_off(mr) + 4 * (kMaxRows + 2); }
static_assert(kMaxCluster * kMaxRows * kRowsCta * 4 + 256 <= tab_bytes(1), "slice sums fit the table area");
static_assert(kThreads * 4 + 4 + 256 <= tab_bytes(1), "the bad-id list fits the table area");
static_assert(32 * kPairBytes <= kTabBlock && 31 * kPairBytes + 256 <= kTabBlock, "pairs fit a block");

// Offset of the 256-byte aligned table area from the dynamic shared memory.
__device__ __forceinline__ uint32_t tab_align(uint32_t sbase) { return (256u - (sbase & 255u)) & 255u; }

struct Params {
  const float* x;
  const uint8_t* w;
  float* y;
  const int32_t* ids;
  int* flags;
  int M, row0;  // plain calls: activation rows row0 .. row0 + M - 1
  int N, K, nb, tiles, rgroups;
  int ks, bps;         // CTAs of a cluster (K slices) and blocks per slice
  long long wstride;   // bytes per expert
  int T, E;            // routed
  int prefetch;        // request the first records before waiting for earlier kernels
  int spc, csz;        // K slices per CTA (1 .. kMaxSpc) and CTAs per cluster (ceil(ks / spc))
};

// bf16 bits of lane l of a group with code c and sign bit s (the row gather).
__device__ uint32_t lane_bf16(int c, int s, int l) {
  const int zero = c >> 2;
  if (l == zero) return 0u;
  const int rank = l - (l > zero ? 1 : 0);  // place among the three other lanes
  const int flip = rank == 0 ? (c & 1) : rank == 1 ? ((c >> 1) & 1) : 0;
  return (flip ^ s) ? 0xBF80u : 0x3F80u;
}

__device__ __forceinline__ uint2 lds64u(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t word4(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Byte offsets in a pair of groups (4 * label, label = code | sign << 4,
// plus 128 for the odd group) of the 8 groups of one code word: `even` holds
// groups 0, 2, 4, 6 in bytes 0..3, `odd` groups 1, 3, 5, 7; s8 has the sign
// of group k at bit k.  The multiply moves sign bits 0, 2, 4, 6 to bits 6,
// 14, 22, 30 (its other partial products land elsewhere and are masked off).
__device__ __forceinline__ void labels8(uint32_t w, uint32_t s8, uint32_t& even, uint32_t& odd) {
  constexpr uint32_t kSpread = 0x01041040u;
  even = ((w << 2) & 0x3C3C3C3Cu) | (((s8 & 0x55u) * kSpread) & 0x40404040u);
  odd = ((w >> 2) & 0x3C3C3C3Cu) | ((((s8 >> 1) & 0x55u) * kSpread) & 0x40404040u) | 0x80808080u;
}

// The table of one chunk of blocks (cb .. ce - 1) for activation rows
// tok[0 .. mrows): MR * tab_blocks(MR) * 64 = 512 (row, group) items, at most
// two per thread.  Their activations are loaded (xload) while the previous
// chunk's lookups run, then turned into entries (layout: tab_row_bytes).
constexpr int kItems = 512 / kThreads;

template <int MR>
__device__ __forceinline__ void xload(const Params& p, const int* tok, int mrows, int cb, int ce,
                                      float (&xl)[kItems][4]) {
  const int groups = (ce - cb) * 64, items = mrows * groups;
#pragma unroll
  for (int u = 0; u < kItems; ++u) {
    const int it = (int)threadIdx.x + u * kThreads;
    if (it < items) {
      const int m = it / groups, gi = it - m * groups;
      const int b = cb + (gi >> 6), g = gi & 63;
      const float* xs = p.x + (long long)tok[m] * p.K + b * kBlockW + (g >> 4) * 64 + (g & 15);
#pragma unroll
      for (int l = 0; l < 4; ++l) xl[u][l] = __ldg(xs + 16 * l);
    }
  }
}

template <int MR>
__device__ __forceinline__ void build_table(uint8_t* tab, int mrows, int cb, int ce, const float (&xl)[kItems][4]) {
  const int groups = (ce - cb) * 64, items = mrows * groups;
#pragma unroll
  for (int u = 0; u < kItems; ++u) {
    const int it = (int)threadIdx.x + u * kThreads;
    if (it >= items) continue;
    const int m = it / groups, gi = it - m * groups;
    float* t = reinterpret_cast<float*>(tab + m * tab_row_bytes(MR) + (gi >> 6) * kTabBlock +
                                        ((gi & 63) >> 1) * kPairBytes + (gi & 1) * 128);
    // The two groups of a pair lie 128 bytes (32 banks) apart, so an odd
    // group's thread writes its sign-set half first: the two stores of a
    // pair then go to banks 16 apart instead of to the same bank.
    const int sw = (gi & 1) * 16;
    const uint32_t sgn = (uint32_t)sw << 27;  // the sign bit for the odd groups' first stores
#pragma unroll
    for (int z = 0; z < 4; ++z) {  // the zero lane; p < q < r the others
      const float xp = xl[u][z == 0 ? 1 : 0], xq = xl[u][z <= 1 ? 2 : 1], xr = xl[u][z <= 2 ? 3 : 2];
      const float uu = __fadd_rn(xr, xq), v = __fsub_rn(xr, xq);
      const float e[4] = {__fadd_rn(uu, xp), __fsub_rn(uu, xp), __fadd_rn(v, xp), __fsub_rn(v, xp)};
#pragma unroll
      for (int f = 0; f < 4; ++f) {  // code 4z + f: bit 0 negates lane p, bit 1 lane q; + 16: all negated
        const uint32_t a = __float_as_uint(e[f]) ^ sgn;
        t[4 * z + f + sw] = __uint_as_float(a);
        t[4 * z + f + 16 - sw] = __uint_as_float(a ^ 0x80000000u);
      }
    }
  }
}

// One block of this lane's row: the 64 groups' entries of every activation
// row summed as (s_0 + s_1) + (s_2 + s_3), s_i over the groups i (mod 4).
// `base` (256-byte aligned) addresses the block in activation row 0's table.
template <int MR>
__device__ __forceinline__ void block_sums(const uint4& c0, const uint4& c1, const uint2& sg, uint32_t base,
                                           float (&bsum)[MR]) {
  float ch[MR][4];
#pragma unroll
  for (int wi = 0; wi < 8; ++wi) {
    const uint32_t w = wi < 4 ? word4(c0, wi) : word4(c1, wi - 4);
    const uint32_t s8 = ((wi < 4 ? sg.x : sg.y) >> (8 * (wi & 3))) & 0xFFu;
    uint32_t lab[2];
    labels8(w, s8, lab[0], lab[1]);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int g = 8 * wi + k;  // byte k >> 1 of lab[k & 1]; pair g >> 1
      const uint32_t a = __byte_perm(lab[k & 1], base, 0x7650u | (uint32_t)(k >> 1));
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        const float v = lds_f32(a + (uint32_t)((g >> 1) * kPairBytes + m * tab_row_bytes(MR)));
        ch[m][g & 3] = g < 4 ? v : __fadd_rn(ch[m][g & 3], v);
      }
    }
  }
#pragma unroll
  for (int m = 0; m < MR; ++m) bsum[m] = __fadd_rn(__fadd_rn(ch[m][0], ch[m][1]), __fadd_rn(ch[m][2], ch[m][3]));
}

// The (up to MR) activation rows of one pass over this CTA's 256 weight rows
// and K slice; the slice sums go to the first CTA of the cluster, which adds
// them in slice order and writes y.  Returns false when a record wait ran out.
// MULTI: the CTA may take several K slices (p.spc > 1; routed calls).
template <int MR, bool MULTI>
__device__ bool run_pass(const Params& p, const uint8_t* wmat, uint8_t* smem, const int* tok, int mrows, int rank,
                         int rg, uint32_t& issued, uint32_t& consumed, uint64_t pol, bool requested) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t talign = tab_align(sbase);
  uint8_t* tab = smem + talign;  // 256-byte aligned
  float* part = reinterpret_cast<float*>(tab);
  const uint32_t ring = sbase + ring_off(MR) + warp * kDepth * kSlot;
  const uint32_t bars = sbase + bar_off(MR) + warp * kDepth * 8;
  const int row_w = rg * kRowsCta + 32 * warp;  // the warp's first weight row
  const int tile0 = row_w >> 4;
  const int ntiles = row_w < p.N ? min(2, p.tiles - tile0) : 0;
  const int half = lane >> 4, r16 = lane & 15;
  const bool lane_rec = half < ntiles;  // the lane's record exists (rows past N in it are zero)
  // this CTA's K slices s0 .. s1 - 1 and their blocks
  const int s0 = rank * p.spc, s1 = min(p.ks, s0 + p.spc);
  const int b0 = s0 * p.bps, b1 = min(p.nb, s1 * p.bps);
  bool ok = true;

  // lane 0 requests block b into the next slot; every lane counts it
  auto request = [&](int b) {
    if (lane == 0) {
      const uint32_t slot = issued % kDepth, bar = bars + 8 * slot, dst = ring + slot * kSlot;
      mbar_expect_tx(bar, (uint32_t)(ntiles * kRec));
      for (int t = 0; t < ntiles; ++t)
        bulk_load(dst + t * kRec, wmat + ((long long)(tile0 + t) * p.nb + b) * kRec, kRec, bar, pol);
    }
    ++issued;
  };
  // the first kDepth blocks: requested here, or before the wait for earlier
  // kernels (`requested`)
  int next_b = min(b1, b0 + kDepth);
  if (ntiles > 0 && !requested) {
    if (lane == 0) fence_proxy_async();
    for (int b = b0; b < next_b; ++b) request(b);
  }

  // acc: the current slice's sum.  The first CTA of a cluster folds its
  // finished slices' sums in slice order (fold); the others keep each one
  // (sl) for the first CTA to fold in after its own.
  constexpr int SPC = MULTI ? kMaxSpc : 1;
  float acc[MR], fold[MR], sl[SPC][MR];
#pragma unroll
  for (int m = 0; m < MR; ++m) {
    acc[m] = fold[m] = 0.f;
#pragma unroll
    for (int j = 0; j < SPC; ++j) sl[j][m] = 0.f;
  }
  auto slice_done = [&](int j) {  // local slice j (0 .. spc - 1) has ended
    if (rank == 0) {
#pragma unroll
      for (int m = 0; m < MR; ++m) fold[m] = j == 0 ? acc[m] : __fadd_rn(fold[m], acc[m]);
    } else {
#pragma unroll
      for (int jj = 0; jj < SPC; ++jj)
#pragma unroll
        for (int m = 0; m < MR; ++m)
          if (jj == j) sl[jj][m] = acc[m];
    }
#pragma unroll
    for (int m = 0; m < MR; ++m) acc[m] = 0.f;
  };
  float xl[kItems][4];
  xload<MR>(p, tok, mrows, b0, min(b1, b0 + tab_blocks(MR)), xl);
  int slice_end = b0 + p.bps;  // MULTI: the first block of the next slice
  for (int cb = b0; cb < b1; cb += tab_blocks(MR)) {
    const int ce = min(b1, cb + tab_blocks(MR));
    __syncthreads();  // the previous chunk's lookups are done
    build_table<MR>(tab, mrows, cb, ce, xl);
    __syncthreads();
    if (ce < b1) xload<MR>(p, tok, mrows, ce, min(b1, ce + tab_blocks(MR)), xl);  // in flight during the lookups
    if (ntiles == 0) continue;
    for (int b = cb; b < ce && ok; ++b) {
      const uint32_t slot = consumed % kDepth, parity = (consumed / kDepth) & 1u;
      ok = __all_sync(0xffffffffu, mbar_wait(bars + 8 * slot, parity));
      if (!ok) break;
      const uint32_t rec = ring + slot * kSlot + half * kRec;
      uint4 c0 = make_uint4(0u, 0u, 0u, 0u), c1 = c0;
      uint2 sg = make_uint2(0u, 0u);
      uint16_t dh = 0;
      if (lane_rec) {
        c0 = lds128(rec + 16 * r16);
        c1 = lds128(rec + 256 + 16 * r16);
        sg = lds64u(rec + kSignOff + 8 * r16);
        dh = lds16(rec + kScaleOff + 2 * r16);
      }
      ++consumed;
      __syncwarp();  // every lane has read the slot
      if (next_b < b1) {
        if (lane == 0) fence_proxy_async();
        request(next_b++);
      }
      float bsum[MR];
      block_sums<MR>(c0, c1, sg, sbase + talign + (uint32_t)((b - cb) * kTabBlock), bsum);
      const float d = __half2float(__ushort_as_half(dh));
      if (MULTI && b == slice_end) {
        slice_done((b - b0) / p.bps - 1);
        slice_end += p.bps;
      }
#pragma unroll
      for (int m = 0; m < MR; ++m) acc[m] = __fmaf_rn(d, bsum[m], acc[m]);
    }
  }
  slice_done(s1 - 1 - s0);
  if (!ok) {
    // let the copies in flight land before the slots are released
    while (consumed < issued) {
      mbar_wait(bars + 8 * (consumed % kDepth), (consumed / kDepth) & 1u);
      ++consumed;
    }
  }

  // slice sums: [slice][activation row][row of the CTA] in the first CTA's
  // table area; slot 0 holds the first CTA's fold of its slices
  const int row_c = 32 * warp + lane, n = rg * kRowsCta + row_c;
  if (p.csz == 1) {
    if (n < p.N)
#pragma unroll
      for (int m = 0; m < MR; ++m)
        if (m < mrows) p.y[(long long)tok[m] * p.N + n] = fold[m];
    return ok;
  }
  auto to_first = [&](int slice, int m, float v) {
    st_cluster_f32(cluster_map(sbase + talign + 4u * (uint32_t)((slice * kMaxRows + m) * kRowsCta + row_c), 0u), v);
  };
  __syncthreads();  // every warp's table reads are done
  cluster_arrive();
  cluster_wait();  // ... in every CTA of the cluster
  if (n < p.N) {
#pragma unroll
    for (int m = 0; m < MR; ++m) {
      if (m >= mrows) continue;
      if (rank == 0) {
        to_first(0, m, fold[m]);
      } else {
#pragma unroll
        for (int j = 0; j < SPC; ++j)
          if (j < s1 - s0) to_first(s0 + j, m, sl[j][m]);
      }
    }
  }
  cluster_arrive();
  cluster_wait();
  if (rank == 0) {
    for (int o = threadIdx.x; o < mrows * kRowsCta; o += kThreads) {
      const int m = o / kRowsCta, r = o - m * kRowsCta, nn = rg * kRowsCta + r;
      if (nn >= p.N) continue;
      float s = part[m * kRowsCta + r];
      for (int k = p.spc; k < p.ks; ++k) s = __fadd_rn(s, part[(k * kMaxRows + m) * kRowsCta + r]);
      p.y[(long long)tok[m] * p.N + nn] = s;
    }
  }
  return ok;
}

template <int MR, bool ROUTED>
__global__ void __launch_bounds__(kThreads, 2) stq1_tab_kernel(const Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_launch_dependents();
  int* tok = reinterpret_cast<int*>(smem + tok_off(MR));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = p.csz > 1 ? (int)cluster_rank() : 0;
  const int rg = (int)blockIdx.x / p.csz;
  const int e = ROUTED ? (int)blockIdx.y : 0;
  const uint8_t* wmat = p.w + (long long)e * p.wstride;
  const uint64_t pol = policy_evict_first();

  if (lane == 0)
    for (int i = 0; i < kDepth; ++i) mbar_init(smem_u32(smem) + bar_off(MR) + (warp * kDepth + i) * 8, 1);
  fence_barrier_init();
  uint32_t issued = 0, consumed = 0;
  // The weights never depend on earlier kernels: in plain mode the first
  // records are requested before the wait for those kernels; activations,
  // ids and outputs are only touched after it.
  const bool early = !ROUTED && p.prefetch;
  if (early) {
    const int row_w = rg * kRowsCta + 32 * warp, tile0 = row_w >> 4;
    const int ntiles = row_w < p.N ? min(2, p.tiles - tile0) : 0;
    const int b0 = rank * p.spc * p.bps, b1 = min(p.nb, (rank + 1) * p.spc * p.bps);
    for (int b = b0; b < b1 && b < b0 + kDepth && ntiles > 0; ++b) {
      if (lane == 0) {
        const uint32_t slot = issued % kDepth;
        const uint32_t bar = smem_u32(smem) + bar_off(MR) + (warp * kDepth + slot) * 8;
        const uint32_t dst = smem_u32(smem) + ring_off(MR) + (warp * kDepth + slot) * kSlot;
        mbar_expect_tx(bar, (uint32_t)(ntiles * kRec));
        for (int t = 0; t < ntiles; ++t)
          bulk_load(dst + t * kRec, wmat + ((long long)(tile0 + t) * p.nb + b) * kRec, kRec, bar, pol);
      }
      ++issued;
    }
  }
  pdl_wait();
  if (ROUTED && blockIdx.x == 0 && blockIdx.y == 0) {
    // tokens routed outside 0..E-1: zero rows and the device flag.  The ids
    // are checked a CTA's width at a time (one thread per token), the bad
    // ones listed in shared memory, and their rows zeroed by every thread.
    int* s_bad = reinterpret_cast<int*>(smem);  // the table area, not in use yet
    int& s_nbad = s_bad[kThreads];
    for (int t0 = 0; t0 < p.T; t0 += kThreads) {
      if (threadIdx.x == 0) s_nbad = 0;
      __syncthreads();
      const int tt = t0 + (int)threadIdx.x;
      if (tt < p.T) {
        const int id = __ldg(p.ids + tt);
        if (id < 0 || id >= p.E) s_bad[atomicAdd(&s_nbad, 1)] = tt;
      }
      __syncthreads();
      const int nbad = s_nbad;
      if (nbad > 0 && threadIdx.x == 0) atomicOr(p.flags, W4A16_DEVICE_BAD_ID);
      for (long long i = threadIdx.x; i < (long long)nbad * p.N; i += kThreads)
        p.y[(long long)s_bad[i / p.N] * p.N + i % p.N] = 0.f;
      __syncthreads();
    }
  }
  bool ok = true;
  int next = 0;  // routed: first token not yet gathered
  for (;;) {
    int mrows;
    __syncthreads();  // barrier inits; earlier passes are done with tok and the table area
    if (ROUTED) {
      if (warp == 0) {
        int cnt = 0, t0 = next;
        while (cnt < MR && t0 < p.T) {
          const int tt = t0 + lane;
          const bool hit = tt < p.T && __ldg(p.ids + tt) == e;
          const unsigned mask = __ballot_sync(0xFFFFFFFFu, hit);
          const int hits = __popc(mask);
          const int take = min(hits, MR - cnt);
          const int pos = __popc(mask & ((1u << lane) - 1u));
          if (hit && pos < take) tok[cnt + pos] = tt;
          cnt += take;
          if (take < hits) {  // stop at the first hit not taken
            unsigned rest = mask;
            for (int q = 0; q < take; ++q) rest &= rest - 1u;
            t0 += __ffs(rest) - 1;
            break;
          }
          t0 += 32;
        }
        if (lane == 0) {
          tok[kMaxRows] = cnt;
          tok[kMaxRows + 1] = min(t0, p.T);
        }
      }
      __syncthreads();
      mrows = tok[kMaxRows];
      next = tok[kMaxRows + 1];
      if (mrows == 0) break;  // the same in every CTA of the cluster
    } else {
      if ((int)threadIdx.x < p.M) tok[threadIdx.x] = p.row0 + (int)threadIdx.x;
      mrows = p.M;
      __syncthreads();
    }
    ok = run_pass<MR, ROUTED>(p, wmat, smem, tok, mrows, rank, rg, issued, consumed, pol, early) && ok;
    if (!ROUTED) break;
  }
  if (!ok && lane == 0 && p.flags) atomicOr(p.flags, W4A16_DEVICE_TIMEOUT);
}

// ---- repack and row gather -----------------------------------------------------------

__global__ void stq1_pack_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int N, int nb,
                                 int tiles) {
  const long long total = (long long)tiles * 16 * nb;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int b = (int)(i % nb);
    const long long row = i / nb;
    const int r = (int)(row & 15);
    uint8_t* rec = dst + ((row >> 4) * nb + b) * kRec;
    uint16_t h[21];
    if (row < N) {
      const uint16_t* s16 = reinterpret_cast<const uint16_t*>(src + (row * nb + b) * kBlockBytes);
#pragma unroll
      for (int q = 0; q < 21; ++q) h[q] = s16[q];
    } else {
#pragma unroll
      for (int q = 0; q < 21; ++q) h[q] = 0;
    }
    uint16_t* c0 = reinterpret_cast<uint16_t*>(rec + 16 * r);        // qs bytes 0..15
    uint16_t* c1 = reinterpret_cast<uint16_t*>(rec + 256 + 16 * r);  // qs bytes 16..31
    uint16_t* sg = reinterpret_cast<uint16_t*>(rec + kSignOff + 8 * r);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      c0[q] = h[q];
      c1[q] = h[8 + q];
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) sg[q] = h[16 + q];
    *reinterpret_cast<uint16_t*>(rec + kScaleOff + 2 * r) = h[20];
  }
}

// out[t][k] = W[ids[t]][k]; one thread per (token, block, group).
__global__ void stq1_rows_kernel(const uint8_t* __restrict__ w, const int32_t* __restrict__ ids,
                                 float* __restrict__ out, int T, int N, int K, int nb, int* flags) {
  const long long total = (long long)T * nb * 64;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int g = (int)(i & 63), tq = g >> 4, j = g & 15;
    const long long rest = i >> 6;
    const int b = (int)(rest % nb);
    const long long t = rest / nb;
    float* o = out + t * K + b * kBlockW + tq * 64 + j;
    const int n = __ldg(ids + t);
    if (n < 0 || n >= N) {
      if (b == 0 && g == 0) atomicOr(flags, W4A16_DEVICE_BAD_ID);
      o[0] = o[16] = o[32] = o[48] = 0.f;
      continue;
    }
    const int r = n & 15;
    const uint8_t* rec = w + ((long long)(n >> 4) * nb + b) * kRec;
    const int code = (rec[256 * (g >> 5) + 16 * r + ((g & 31) >> 1)] >> (4 * (g & 1))) & 15;
    const int s = (rec[kSignOff + 8 * r + (g >> 3)] >> (g & 7)) & 1;
    const float d =
        __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(rec + kScaleOff + 2 * r)));
#pragma unroll
    for (int q = 0; q < 4; ++q) o[16 * q] = d * __uint_as_float(lane_bf16(code, s, q) << 16);
  }
}

// ---- host side -------------------------------------------------------------------------

template <int MR, bool ROUTED>
cudaError_t launch_tab(const Params& p, int pdl, cudaStream_t s) {
  auto fn = stq1_tab_kernel<MR, ROUTED>;
  static std::mutex mu;
  static std::map<int, bool> ready;  // device -> shared-memory attribute set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!ready[dev]) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes(MR));
      if (e != cudaSuccess) return e;
      ready[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(p.csz * p.rgroups), ROUTED ? (unsigned)p.E : 1u, 1u);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem_bytes(MR);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  unsigned n = 0;
  if (p.csz > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)p.csz;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl > 0) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, fn, p);
}

template <bool ROUTED>
cudaError_t launch_rows(const Params& p, int MR, int pdl, cudaStream_t s) {
  switch (MR) {
    case 1: return launch_tab<1, ROUTED>(p, pdl, s);
    case 2: return launch_tab<2, ROUTED>(p, pdl, s);
    case 4: return launch_tab<4, ROUTED>(p, pdl, s);
    case 8: return launch_tab<8, ROUTED>(p, pdl, s);
    default: return cudaErrorInvalidValue;
  }
}

Params base_params(int N, int K) {
  Stq1Plan pl;
  stq1_make_plan(N, K, &pl);
  Params p{};
  p.N = N;
  p.K = K;
  p.nb = pl.nb;
  p.tiles = pl.tiles;
  p.rgroups = pl.rgroups;
  p.ks = pl.ks;
  p.bps = pl.bps;
  p.spc = 1;  // one K slice per CTA: a cluster of ks CTAs per row group
  p.csz = pl.ks;
  p.wstride = (long long)stq1_packed_size(N, K);
  return p;
}

int pow2_at_least(int v) {
  int r = 1;
  while (r < v) r *= 2;
  return r;
}

}  // namespace

bool stq1_shape_ok(int N, int K) { return N >= 1 && K >= kBlockW && K <= 32768 && K % kBlockW == 0; }

size_t stq1_packed_size(int N, int K) {
  if (!stq1_shape_ok(N, K)) return 0;
  return (size_t)((N + 15) / 16) * (size_t)(K / kBlockW) * kRec;
}

void stq1_make_plan(int N, int K, Stq1Plan* pl) {
  pl->nb = K / kBlockW;
  pl->tiles = (N + 15) / 16;
  pl->rgroups = (N + kRowsCta - 1) / kRowsCta;
  // K slices: as many as keep the grid within one wave of resident CTAs, at
  // most a portable cluster and one block per slice; then as few slices as
  // that slice length needs
  int ks = kWaveCtas / pl->rgroups;
  ks = std::max(1, std::min(ks, std::min(kMaxCluster, pl->nb)));
  pl->bps = (pl->nb + ks - 1) / ks;
  pl->ks = (pl->nb + pl->bps - 1) / pl->bps;
  pl->xcap = kMaxRows;
}

cudaError_t launch_stq1_pack(const uint8_t* src, uint8_t* dst, int N, int K, cudaStream_t s) {
  const int nb = K / kBlockW, tiles = (N + 15) / 16;
  const long long total = (long long)tiles * 16 * nb;
  long long blocks = (total + 255) / 256;
  if (blocks > 65535) blocks = 65535;
  stq1_pack_kernel<<<(unsigned)blocks, 256, 0, s>>>(src, dst, N, nb, tiles);
  return cudaGetLastError();
}

cudaError_t launch_stq1_mm(const float* x, const uint8_t* w, float* y, int M, int row0, int N, int K, int* flags,
                           int pdl, cudaStream_t s) {
  Params p = base_params(N, K);
  if (M < 1 || M > kMaxRows) return cudaErrorInvalidValue;
  p.flags = flags;
  p.prefetch = pdl >= 2;
  p.x = x;
  p.w = w;
  p.y = y;
  p.M = M;
  p.row0 = row0;
  return launch_rows<false>(p, pow2_at_least(M), pdl, s);
}

cudaError_t launch_stq1_mm_id(const float* x, const uint8_t* w, const int32_t* ids, float* y, int T, int N,
                              int K, int E, int* flags, int pdl, cudaStream_t s) {
  Params p = base_params(N, K);
  p.x = x;
  p.w = w;
  p.y = y;
  p.ids = ids;
  p.flags = flags;
  p.T = T;
  p.E = E;
  // Routed calls touch many experts: each CTA takes up to kMaxSpc K slices
  // of its rows (the same slice sums, folded in the same order), so the grid
  // has fewer, longer CTAs per expert.
  p.spc = std::min(p.ks, kMaxSpc);
  p.csz = (p.ks + p.spc - 1) / p.spc;
  // Tokens per pass: twice the mean per expert (at least two), at most T and
  // eight; an expert with more tokens takes more passes.
  long long want = 2LL * ((T + E - 1) / E);
  if (want < 2) want = 2;
  if (want > T) want = T;
  int R = pow2_at_least((int)want);
  if (R > kMaxRows) R = kMaxRows;
  return launch_rows<true>(p, R, pdl, s);
}

cudaError_t launch_stq1_get_rows(const uint8_t* w, const int32_t* ids, float* out, int T, int N, int K,
                                 int* flags, cudaStream_t s) {
  const int nb = K / kBlockW;
  const long long total = (long long)T * nb * 64;
  long long blocks = (total + 255) / 256;
  if (blocks > 65535) blocks = 65535;
  stq1_rows_kernel<<<(unsigned)blocks, 256, 0, s>>>(w, ids, out, T, N, K, nb, flags);
  return cudaGetLastError();
}

}  // namespace w4a16

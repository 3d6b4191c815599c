// stq1.cu -- the STQ1_0 ternary matmul on the tensor cores (sm_103a).
//
// "Hy4-preview Metal kernels for llama.cpp" gives the format (section "Notes
// and gotchas": 42-byte blocks of 256 weights, 4-bit group codes, group sign
// bits, an fp16 scale, and the weight-to-group map), the kernels a model
// needs (the kernel table: matvec, small batches, routed experts, row
// gather) and the structure of a group (section "Results", the fourth decode
// pass: one zero lane named by the code's high bits, two sign flips in its
// low bits, the sign bit negating the group).  The Metal schedule itself is
// not the design here:
//
//  * Weights keep the page's 42 bytes per 256, repacked once (stq1_pack) into
//    672-byte records per 16-row tile and block, so each lane loads its codes,
//    sign bits and scales with one 16-, one 4- and one 4-byte load.
//  * The contraction runs on the tensor cores (mma.sync m16n8k16, bf16 in,
//    fp32 accumulate).  Ternary lanes are exact in bf16; x enters as three
//    bf16 parts h0 + h1 + h2 = x, each the previous residual truncated to
//    its top 8 significant bits (exact for every finite |x| >= 2^-110: the
//    lowest significand bit then sits at 2^-133 or above, the smallest bf16
//    step; below that the parts lose at most 2^-133), as three columns of
//    B, so the products are exact and only the fp32 accumulation rounds.  Within a block the MMA k
//    order is chosen so that each lane's A fragment holds whole groups: k
//    position 2t+i of chunk j is lane i of group 16t + j, position 2t+8+i is
//    lane 2+i; lane t of a quad then owns groups 16t .. 16t+15, eight
//    contiguous code bytes and sixteen contiguous sign bits of the page's
//    own block.  B follows the same order (the activations are staged in it).
//  * A group decodes through a 32-entry table in shared memory (code and
//    sign bit -> the bf16 pairs of lanes 0,1 and 2,3), one 8-byte slot per
//    warp lane so that lookups never conflict.  The page found a table
//    lookup faster than arithmetic decoding on its GPU; here it also keeps
//    the decode at a few instructions per group: the table offsets of 16
//    groups come from four word-wide mask/multiply steps and one byte
//    permute per group.
//  * Each CTA stages the activation parts once; its 8 warps take K slices of
//    one to eight 16-row tiles per round, add their fp32 partials in shared
//    memory in slice order, and write y.  The slice count and every order
//    depend on (N, K) only, so any row of a multi-row call equals the
//    one-row call bit for bit.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "stq1.cuh"
#include "w4a16.h"

namespace w4a16 {
namespace {

constexpr int kBlockW = 256;     // weights per block
constexpr int kBlockBytes = 42;  // bytes per block in the page's layout
constexpr int kRec = 672;        // bytes per (16-row tile, block) record
constexpr int kSignOff = 512;
constexpr int kScaleOff = 640;
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kDepth = 4;                 // records in flight per warp
constexpr int kMaxRows = 8;               // activation rows per pass
constexpr int kTokBytes = 192;            // int tok[8], count, next token; 32-word expert bitmap
constexpr int kSmemCap = 227 * 1024 - 32 * 32 * 8;  // dynamic share; the decode table is static
constexpr int kSlack = 256;                          // spare bytes after the staged rows
constexpr int kTargetWarps = 2432;        // 152 SMs x 16 warps
constexpr int kGroupStride = 4096;        // staged bytes per block and 8 columns

__host__ __device__ constexpr int red_bytes(int mc) { return kWarps * 16 * 8 * mc * 4; }
__host__ __device__ constexpr int fixed_smem(int mc) { return 2 * red_bytes(mc) + kTokBytes + kSlack; }

struct Params {
  const float* x;
  const uint8_t* w;
  float* y;
  const int32_t* ids;
  int* flags;
  int M, row0;  // plain calls: rows row0 .. row0 + M - 1
  int N, K, nb, tiles;
  int ks, bps, rt, rounds;
  int xcap;
  long long wstride;  // bytes per expert
  int T, E;
  int flat;  // routed: deal (expert, round) units over one grid (E <= 1024)
};

__device__ __forceinline__ uint32_t ld_nc_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// bf16 bits of lane l of a group with code c and sign bit s.
__device__ uint32_t lane_bf16(int c, int s, int l) {
  const int zero = c >> 2;
  if (l == zero) return 0u;
  const int rank = l - (l > zero ? 1 : 0);  // place among the three other lanes
  const int flip = rank == 0 ? (c & 1) : rank == 1 ? ((c >> 1) & 1) : 0;
  return (flip ^ s) ? 0xBF80u : 0x3F80u;
}

// Decode table: the bf16 pairs (lanes 0,1 | lanes 2,3) of label = code | sign << 4,
// one 8-byte copy per warp lane at byte label * 256 + lane * 8, so the 32
// lookups of a warp fall in distinct banks whatever the labels.
__shared__ uint2 s_lut[32 * 32];

__device__ void fill_lut() {
  for (int i = threadIdx.x; i < 32 * 32; i += blockDim.x) {
    const int label = i >> 5, c = label & 15, s = label >> 4;
    s_lut[i] = make_uint2(lane_bf16(c, s, 0) | (lane_bf16(c, s, 1) << 16),
                          lane_bf16(c, s, 2) | (lane_bf16(c, s, 3) << 16));
  }
}

__device__ __forceinline__ uint2 lut_entry(uint32_t byte_offset) {
  return *reinterpret_cast<const uint2*>(reinterpret_cast<const char*>(s_lut) + byte_offset);
}

// Columns of a pass of up to R activation rows: 3R parts, in MMA groups of 8.
template <int R>
struct Cols {
  static constexpr int NC = 3 * R;
  static constexpr int MC = (NC + 7) / 8;
  __host__ __device__ static constexpr int ncg(int g) { return NC - 8 * g < 8 ? NC - 8 * g : 8; }
};

// Activation rows tok[0 .. mrows) of x as bf16 parts in MMA fragment order.
// Column c = 3m + q (part q of row m) is column n = c % 8 of MMA group
// g = c / 8.  Group g occupies `gstride` bytes from g * gstride; in it the
// 8-byte slot of (block b, chunk j, column n, quad lane t) is at
// ((b*16 + j) * ncg(g) + n) * 32 + t * 8 and holds the parts of
// x[256b + 64t + 16p + j], p = 0..3 (lanes 0..3 of group 16t + j): the two
// B registers of that lane.  Each thread loads the four values of a slot
// for four slots before converting any (sixteen loads in flight).
template <int R>
__device__ void stage_rows(uint8_t* bsm, const float* __restrict__ x, const int* tok, int mrows, int K, int nb,
                           int gstride) {
  using C = Cols<R>;
  const int per_row = nb * 64;
  const int total = mrows * per_row;
  for (int base = threadIdx.x; base < total; base += 4 * kThreads) {
    float v[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int it = base + u * kThreads;
      if (it < total) {
        const int m = it / per_row, w = it - m * per_row;
        const float* src = x + (long long)tok[m] * K + (w >> 6) * kBlockW + ((w >> 4) & 3) * 64 + (w & 15);
#pragma unroll
        for (int q = 0; q < 4; ++q) v[u][q] = __ldg(src + 16 * q);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int it = base + u * kThreads;
      if (it < total) {
        const int m = it / per_row, w = it - m * per_row;
        const int b = w >> 6, t = (w >> 4) & 3, j = w & 15;
        uint32_t part[3][2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t bits[3][2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            // each part is the previous residual truncated to its top 16
            // bits (a bf16 with the residual's sign and exponent), so no part
            // rounds up and overflows, and every subtraction is exact
            const float f = v[u][2 * h + e];
            const uint32_t b0 = __float_as_uint(f) & 0xFFFF0000u;
            const float r1 = __fsub_rn(f, __uint_as_float(b0));
            const uint32_t b1 = __float_as_uint(r1) & 0xFFFF0000u;
            const float r2 = __fsub_rn(r1, __uint_as_float(b1));
            bits[0][e] = b0 >> 16;
            bits[1][e] = b1 >> 16;
            bits[2][e] = __float_as_uint(r2) >> 16;
          }
#pragma unroll
          for (int q = 0; q < 3; ++q) part[q][h] = bits[q][0] | (bits[q][1] << 16);
        }
#pragma unroll
        for (int q = 0; q < 3; ++q) {
          const int c = 3 * m + q, g = c >> 3, n = c & 7;
          const int ncg = g < C::MC - 1 ? 8 : C::ncg(C::MC - 1);
          *reinterpret_cast<uint2*>(bsm + g * gstride + ((b * 16 + j) * ncg + n) * 32 + t * 8) =
              make_uint2(part[q][0], part[q][1]);
        }
      }
    }
  }
}

struct Rec {
  uint4 c;     // codes: rows r (x, y) and r + 8 (z, w), 16 groups each
  uint32_t s;  // sign bits: row r (low half), row r + 8 (high half)
  uint32_t d;  // fp16 scales: row r (low), row r + 8 (high)
};

// Table offsets (label * 256, label = code | sign << 4, one byte each) of the
// 16 groups of one row: L[0] groups 0,2,4,6; L[1] 1,3,5,7; L[2] 8,..,14;
// L[3] 9,..,15.  The multiply moves sign bits 0, 2, 4, 6 to bits 4, 12, 20,
// 28 (its other partial products land elsewhere and are masked off).
__device__ __forceinline__ void labels(uint32_t lo, uint32_t hi, uint32_t sg, uint32_t L[4]) {
  constexpr uint32_t kSpread = 0x00410410u;
  L[0] = (lo & 0x0F0F0F0Fu) | (((sg & 0x55u) * kSpread) & 0x10101010u);
  L[1] = ((lo >> 4) & 0x0F0F0F0Fu) | ((((sg >> 1) & 0x55u) * kSpread) & 0x10101010u);
  L[2] = (hi & 0x0F0F0F0Fu) | ((((sg >> 8) & 0x55u) * kSpread) & 0x10101010u);
  L[3] = ((hi >> 4) & 0x0F0F0F0Fu) | ((((sg >> 9) & 0x55u) * kSpread) & 0x10101010u);
}

__device__ __forceinline__ void mma_bf16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One record (block b of a 16-row tile): 16 chunks of 16 k, one MMA per
// active column group (even and odd chunks in two accumulators), then
// pa += d * (even + odd) per row.  Lanes whose column
// lies past a group's last one read that last column's slot again (a
// broadcast: no extra shared-memory traffic); those columns of C are never
// used.
template <int R>
__device__ __forceinline__ void process(const Rec& r, const uint8_t* bsm, int b, int gstride, int active_groups,
                                        uint32_t lane8, int n, int t, float pa[Cols<R>::MC][4]) {
  using C = Cols<R>;
  uint32_t La[4], Lb[4];
  labels(r.c.x, r.c.y, r.s & 0xFFFFu, La);
  labels(r.c.z, r.c.w, r.s >> 16, Lb);
  const uint2* bq[C::MC];
  float acc[2][C::MC][4];  // even and odd chunks: two shorter MMA dependency chains
#pragma unroll
  for (int g = 0; g < C::MC; ++g) {
    const int col = n < C::ncg(g) ? n : C::ncg(g) - 1;
    bq[g] = reinterpret_cast<const uint2*>(bsm + g * gstride + (b * 16 * C::ncg(g) + col) * 32 + t * 8);
#pragma unroll
    for (int h = 0; h < 2; ++h) acc[h][g][0] = acc[h][g][1] = acc[h][g][2] = acc[h][g][3] = 0.f;
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int wi = (j & 1) + 2 * (j >> 3);
    const uint32_t sel = 0x5504u | ((uint32_t)((j >> 1) & 3) << 4);  // [0, 0, label, lane8]
    const uint2 ea = lut_entry(__byte_perm(La[wi], lane8, sel));
    const uint2 eb = lut_entry(__byte_perm(Lb[wi], lane8, sel));
#pragma unroll
    for (int g = 0; g < C::MC; ++g) {
      if (g == 0 || g < active_groups) {
        const uint2 bf = bq[g][j * C::ncg(g) * 4];
        mma_bf16(acc[j & 1][g], ea.x, eb.x, ea.y, eb.y, bf.x, bf.y);
      }
    }
  }
  const float dr = __half2float(__ushort_as_half((unsigned short)(r.d & 0xFFFFu)));
  const float dr8 = __half2float(__ushort_as_half((unsigned short)(r.d >> 16)));
#pragma unroll
  for (int g = 0; g < C::MC; ++g) {
    pa[g][0] = __fmaf_rn(dr, __fadd_rn(acc[0][g][0], acc[1][g][0]), pa[g][0]);
    pa[g][1] = __fmaf_rn(dr, __fadd_rn(acc[0][g][1], acc[1][g][1]), pa[g][1]);
    pa[g][2] = __fmaf_rn(dr8, __fadd_rn(acc[0][g][2], acc[1][g][2]), pa[g][2]);
    pa[g][3] = __fmaf_rn(dr8, __fadd_rn(acc[0][g][3], acc[1][g][3]), pa[g][3]);
  }
}

// End of a round: the warps' partials through shared memory (buffer `buf`
// of two, so one barrier per round), summed over the K slices in slice
// order, then the three parts (h0 + h1) + h2, into y.
template <int R>
__device__ void finish_round(const Params& p, float* red, int buf, const int* tok, int mrows, int tile0, int warp,
                             int lane, float pa[Cols<R>::MC][4]) {
  using C = Cols<R>;
  constexpr int stride = 8 * C::MC;
  float* rb = red + buf * (kWarps * 16 * stride);
  const int r = lane >> 2, t = lane & 3;
#pragma unroll
  for (int g = 0; g < C::MC; ++g) {
    *reinterpret_cast<float2*>(rb + (warp * 16 + r) * stride + 8 * g + 2 * t) = make_float2(pa[g][0], pa[g][1]);
    *reinterpret_cast<float2*>(rb + (warp * 16 + r + 8) * stride + 8 * g + 2 * t) = make_float2(pa[g][2], pa[g][3]);
  }
  __syncthreads();
  const int outs = p.rt * mrows * 16;
  for (int o = threadIdx.x; o < outs; o += kThreads) {
    const int rr = o & 15, mo = o >> 4;
    const int lt = mo / mrows, m = mo - lt * mrows;
    const int tile = tile0 + lt;
    const int n = tile * 16 + rr;
    if (tile < p.tiles && n < p.N) {
      float part[3];
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const int col = 3 * m + q;
        float s = rb[(lt * p.ks * 16 + rr) * stride + col];
        for (int sl = 1; sl < p.ks; ++sl) s = __fadd_rn(s, rb[((lt * p.ks + sl) * 16 + rr) * stride + col]);
        part[q] = s;
      }
      p.y[(long long)tok[m] * p.N + n] = __fadd_rn(__fadd_rn(part[0], part[1]), part[2]);
    }
  }
}

// The rounds a CTA runs on one matrix: first, first + step, ... (count).
struct Span {
  int first, count, step;
};

// A warp's stream of records: round `first + k * step` of its span (tile
// round * rt + lt), blocks slice * bps .. slice * bps + bps - 1 of each.
struct Cursor {
  const uint8_t* rec;
  int tile, i, tile_step;
};

__device__ __forceinline__ void cursor_start(Cursor& c, const Params& p, const uint8_t* wbase, const Span& sp, int lt,
                                             int slice) {
  c.tile = sp.first * p.rt + lt;
  c.i = 0;
  c.tile_step = sp.step * p.rt;
  c.rec = wbase + ((long long)c.tile * p.nb + slice * p.bps) * kRec;
}

__device__ __forceinline__ bool cursor_valid(const Cursor& c, const Params& p, int slice) {
  return c.tile < p.tiles && slice * p.bps + c.i < p.nb;
}

__device__ __forceinline__ void cursor_next(Cursor& c, const Params& p, const uint8_t* wbase, int slice) {
  if (++c.i == p.bps) {
    c.i = 0;
    c.tile += c.tile_step;
    c.rec = wbase + ((long long)c.tile * p.nb + slice * p.bps) * kRec;
  } else {
    c.rec += kRec;
  }
}

__device__ __forceinline__ void fetch(Cursor& c, const Params& p, const uint8_t* wbase, int slice, int lane,
                                      Rec& r) {
  if (cursor_valid(c, p, slice)) {
    r.c = ld_stream_v4(c.rec + 16 * lane);
    r.s = ld_nc_u32(c.rec + kSignOff + 4 * lane);
    r.d = ld_nc_u32(c.rec + kScaleOff + 4 * (lane >> 2));
  } else {
    r.c = make_uint4(0u, 0u, 0u, 0u);
    r.s = 0u;
    r.d = 0u;
  }
  cursor_next(c, p, wbase, slice);
}

// The rounds of `sp` on one matrix (expert e when routed): passes of at most
// R activation rows (routed: the expert's tokens in order), each staged once,
// then every warp's records of the span.
template <int R, bool ROUTED>
__device__ void run_span(const Params& p, const uint8_t* wbase, int e, const Span& sp, float* red, int* tok,
                         uint8_t* bsm, int warp, int lane, int lt, int slice) {
  using C = Cols<R>;
  const int gstride = p.nb * kGroupStride;
  const int n_items = sp.count * p.bps;
  const uint32_t lane8 = (uint32_t)lane * 8u;
  const int n = lane >> 2, t = lane & 3;
  int next = 0;  // routed: first token not yet gathered
  for (;;) {
    int mrows;
    __syncthreads();  // earlier passes and spans are done with tok and the staged rows
    if (ROUTED) {
      if (warp == 0) {
        int cnt = 0, t0 = next;
        while (cnt < p.xcap && t0 < p.T) {
          const int tt = t0 + lane;
          const bool hit = tt < p.T && __ldg(p.ids + tt) == e;
          const unsigned mask = __ballot_sync(0xFFFFFFFFu, hit);
          const int hits = __popc(mask);
          const int take = min(hits, p.xcap - cnt);
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
      if (mrows == 0) break;
    } else {
      if ((int)threadIdx.x < p.M) tok[threadIdx.x] = p.row0 + (int)threadIdx.x;
      mrows = p.M;
      __syncthreads();
    }
    // weights first: the first records are in flight while the rows are staged
    Cursor fc, cc;
    cursor_start(fc, p, wbase, sp, lt, slice);
    cursor_start(cc, p, wbase, sp, lt, slice);
    Rec ring[kDepth];
#pragma unroll
    for (int s = 0; s < kDepth; ++s) fetch(fc, p, wbase, slice, lane, ring[s]);
    stage_rows<R>(bsm, p.x, tok, mrows, p.K, p.nb, gstride);
    __syncthreads();
    const int active = (3 * mrows + 7) / 8;
    float pa[C::MC][4];
#pragma unroll
    for (int g = 0; g < C::MC; ++g) pa[g][0] = pa[g][1] = pa[g][2] = pa[g][3] = 0.f;
    int buf = 0;
    for (int base = 0; base < n_items; base += kDepth) {
#pragma unroll
      for (int s = 0; s < kDepth; ++s) {
        if (base + s < n_items) {  // the same for every warp of the CTA
          const Rec cur = ring[s];
          fetch(fc, p, wbase, slice, lane, ring[s]);
          if (cursor_valid(cc, p, slice))
            process<R>(cur, bsm, slice * p.bps + cc.i, gstride, active, lane8, n, t, pa);
          if (cc.i == p.bps - 1) {
            finish_round<R>(p, red, buf, tok, mrows, cc.tile - lt, warp, lane, pa);
            buf ^= 1;
#pragma unroll
            for (int g = 0; g < C::MC; ++g) pa[g][0] = pa[g][1] = pa[g][2] = pa[g][3] = 0.f;
          }
          cursor_next(cc, p, wbase, slice);
        }
      }
    }
    if (!ROUTED) break;
  }
}

// Index of the k-th set bit of a 1024-bit map.
__device__ __forceinline__ int nth_set_bit(const unsigned* bm, int k) {
  for (int w = 0; w < 32; ++w) {
    const int c = __popc(bm[w]);
    if (k < c) {
      unsigned v = bm[w];
      for (int q = 0; q < k; ++q) v &= v - 1u;
      return 32 * w + __ffs(v) - 1;
    }
    k -= c;
  }
  return -1;
}

template <int R, bool ROUTED>
__global__ void __launch_bounds__(kThreads, 2) stq1_mm_kernel(const Params p) {
  using C = Cols<R>;
  extern __shared__ __align__(16) uint8_t smem[];
  float* red = reinterpret_cast<float*>(smem);
  int* tok = reinterpret_cast<int*>(smem + 2 * red_bytes(C::MC));
  unsigned* bitmap = reinterpret_cast<unsigned*>(tok + 16);
  uint8_t* bsm = smem + 2 * red_bytes(C::MC) + kTokBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lt = warp / p.ks, slice = warp - lt * p.ks;
  fill_lut();
  if (!ROUTED) {
    const int mine = (int)blockIdx.x < p.rounds ? (p.rounds - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    run_span<R, false>(p, p.w, 0, Span{(int)blockIdx.x, mine, (int)gridDim.x}, red, tok, bsm, warp, lane, lt, slice);
    return;
  }
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    // tokens routed outside 0..E-1: zero rows and the device flag.  The ids
    // are checked a CTA's width at a time (one thread per token), the bad
    // ones listed in shared memory, and their rows zeroed by every thread.
    int* s_bad = reinterpret_cast<int*>(bsm);  // the activation area, not in use yet
    int& s_nbad = s_bad[kThreads];
    for (int t0 = 0; t0 < p.T; t0 += blockDim.x) {
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
      for (long long i = threadIdx.x; i < (long long)nbad * p.N; i += blockDim.x)
        p.y[(long long)s_bad[i / p.N] * p.N + i % p.N] = 0.f;
      __syncthreads();
    }
  }
  if (!p.flat) {  // one grid column per expert
    const int mine = (int)blockIdx.x < p.rounds ? (p.rounds - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    run_span<R, true>(p, p.w + (long long)blockIdx.y * p.wstride, (int)blockIdx.y,
                      Span{(int)blockIdx.x, mine, (int)gridDim.x}, red, tok, bsm, warp, lane, lt, slice);
    return;
  }
  // One grid over the experts some token selects: units (expert, round) in
  // order, a contiguous range per CTA (at most a few experts each).
  if (threadIdx.x < 32) bitmap[threadIdx.x] = 0u;
  __syncthreads();
  for (int tt = threadIdx.x; tt < p.T; tt += blockDim.x) {
    const int id = __ldg(p.ids + tt);
    if (id >= 0 && id < p.E) atomicOr(&bitmap[id >> 5], 1u << (id & 31));
  }
  __syncthreads();
  int touched = 0;
  for (int w = 0; w < 32; ++w) touched += __popc(bitmap[w]);
  const long long units = (long long)touched * p.rounds;
  long long u = units * blockIdx.x / gridDim.x;
  const long long u_end = units * (blockIdx.x + 1) / gridDim.x;
  while (u < u_end) {
    const int ei = (int)(u / p.rounds);
    const int r = (int)(u - (long long)ei * p.rounds);
    const int cnt = (int)min((long long)(p.rounds - r), u_end - u);
    const int e = nth_set_bit(bitmap, ei);
    run_span<R, true>(p, p.w + (long long)e * p.wstride, e, Span{r, cnt, 1}, red, tok, bsm, warp, lane, lt, slice);
    u += cnt;
  }
}

// ---- repack and row gather -----------------------------------------------------------

__global__ void stq1_pack_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int N, int nb,
                                 int tiles) {
  const long long total = (long long)tiles * 16 * nb;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int b = (int)(i % nb);
    const long long row = i / nb;
    const int r = (int)(row & 15), half = r >> 3, l0 = (r & 7) * 4;
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
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      uint16_t* cd = reinterpret_cast<uint16_t*>(rec + 16 * (l0 + t) + 8 * half);
#pragma unroll
      for (int q = 0; q < 4; ++q) cd[q] = h[4 * t + q];                                       // qs bytes 8t..8t+7
      *reinterpret_cast<uint16_t*>(rec + kSignOff + 4 * (l0 + t) + 2 * half) = h[16 + t];    // sign bytes 2t, 2t+1
    }
    *reinterpret_cast<uint16_t*>(rec + kScaleOff + 4 * (r & 7) + 2 * half) = h[20];          // d
  }
}

// out[t][k] = W[ids[t]][k]; one thread per (token, block, group).
__global__ void stq1_rows_kernel(const uint8_t* __restrict__ w, const int32_t* __restrict__ ids,
                                 float* __restrict__ out, int T, int N, int K, int nb, int* flags) {
  const long long total = (long long)T * nb * 64;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int gq = (int)(i & 63), tq = gq >> 4, j = gq & 15;
    const long long rest = i >> 6;
    const int b = (int)(rest % nb);
    const long long t = rest / nb;
    float* o = out + t * K + b * kBlockW + tq * 64 + j;
    const int n = __ldg(ids + t);
    if (n < 0 || n >= N) {
      if (b == 0 && gq == 0) atomicOr(flags, W4A16_DEVICE_BAD_ID);
      o[0] = o[16] = o[32] = o[48] = 0.f;
      continue;
    }
    const int r = n & 15, half = r >> 3, l = (r & 7) * 4 + tq;
    const uint8_t* rec = w + ((long long)(n >> 4) * nb + b) * kRec;
    const int code = (rec[16 * l + 8 * half + (j >> 1)] >> (4 * (j & 1))) & 15;
    const int s = (rec[kSignOff + 4 * l + 2 * half + (j >> 3)] >> (j & 7)) & 1;
    const float d = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(
        rec + kScaleOff + 4 * (r & 7) + 2 * half)));
#pragma unroll
    for (int q = 0; q < 4; ++q) o[16 * q] = d * __uint_as_float(lane_bf16(code, s, q) << 16);
  }
}

// ---- host side -------------------------------------------------------------------------

// Multiprocessors of the current device (cached per device).
int sm_count() {
  static std::mutex mu;
  static std::map<int, int> cached;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  std::lock_guard<std::mutex> lk(mu);
  auto it = cached.find(dev);
  if (it != cached.end()) return it->second;
  int v = 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 152;
  cached[dev] = v;
  return v;
}

template <int R, bool ROUTED>
cudaError_t launch_kernel(const Params& p, dim3 grid_cap, int smem, cudaStream_t s) {
  auto fn = stq1_mm_kernel<R, ROUTED>;
  static std::mutex mu;
  static std::map<std::pair<int, int>, int> occ;  // (device, smem) -> CTAs per SM
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = occ.find({dev, smem});
    if (it == occ.end()) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemCap);
      if (e != cudaSuccess) return e;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, smem);
      if (e != cudaSuccess) return e;
      if (per_sm < 1) per_sm = 1;
      occ[{dev, smem}] = per_sm;
    } else {
      per_sm = it->second;
    }
  }
  const int slots = per_sm * sm_count();
  dim3 grid = grid_cap;
  if (ROUTED && p.flat) {
    const long long units = (long long)p.E * p.rounds;
    grid.x = (unsigned)(slots < units ? slots : units);
    grid.y = 1;
  } else if (ROUTED) {
    // CTAs per expert: the resident slots over the experts T tokens are
    // expected to touch when drawn uniformly, E (1 - (1 - 1/E)^T).
    double touched = (double)p.E;
    double miss = 1.0;
    for (int t = 0; t < p.T && t < 4096; ++t) miss *= 1.0 - 1.0 / p.E;
    touched *= 1.0 - miss;
    if (touched < 1.0) touched = 1.0;
    int gx = (int)(slots / touched);
    grid.x = (unsigned)(gx < 1 ? 1 : gx < p.rounds ? gx : p.rounds);
  } else {
    grid.x = (unsigned)(slots < p.rounds ? slots : p.rounds);
  }
  fn<<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

Params base_params(int N, int K) {
  Stq1Plan pl;
  stq1_make_plan(N, K, &pl);
  Params p{};
  p.N = N;
  p.K = K;
  p.nb = pl.nb;
  p.tiles = pl.tiles;
  p.ks = pl.ks;
  p.bps = pl.bps;
  p.rt = pl.rt;
  p.rounds = pl.rounds;
  p.xcap = pl.xcap;
  p.wstride = (long long)stq1_packed_size(N, K);
  return p;
}

int pow2_at_least(int v) {
  int r = 1;
  while (r < v) r *= 2;
  return r;
}

int smem_for(int R, int K) { return fixed_smem((3 * R + 7) / 8) + 6 * R * K; }

template <bool ROUTED>
cudaError_t launch_rows(const Params& p, int R, cudaStream_t s) {
  const int smem = smem_for(R, p.K);
  const dim3 grid(1, ROUTED && !p.flat ? (unsigned)p.E : 1u, 1);
  switch (R) {
    case 1: return launch_kernel<1, ROUTED>(p, grid, smem, s);
    case 2: return launch_kernel<2, ROUTED>(p, grid, smem, s);
    case 4: return launch_kernel<4, ROUTED>(p, grid, smem, s);
    case 8: return launch_kernel<8, ROUTED>(p, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
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
  int ks = 1;
  while (ks < kWarps && 2 * ks <= pl->nb && (long long)pl->tiles * ks < kTargetWarps) ks *= 2;
  pl->ks = ks;
  pl->bps = (pl->nb + ks - 1) / ks;
  pl->rt = kWarps / ks;
  pl->rounds = (pl->tiles + pl->rt - 1) / pl->rt;
  // rows per pass: the largest power of two up to 8 whose staged parts fit
  int x = kMaxRows;
  while (x > 1 && smem_for(x, K) > kSmemCap) x /= 2;
  pl->xcap = x;
}

cudaError_t launch_stq1_pack(const uint8_t* src, uint8_t* dst, int N, int K, cudaStream_t s) {
  const int nb = K / kBlockW, tiles = (N + 15) / 16;
  const long long total = (long long)tiles * 16 * nb;
  long long blocks = (total + 255) / 256;
  if (blocks > 65535) blocks = 65535;
  stq1_pack_kernel<<<(unsigned)blocks, 256, 0, s>>>(src, dst, N, nb, tiles);
  return cudaGetLastError();
}

cudaError_t launch_stq1_mm(const float* x, const uint8_t* w, float* y, int M, int row0, int N, int K,
                           cudaStream_t s) {
  Params p = base_params(N, K);
  if (M < 1 || M > p.xcap) return cudaErrorInvalidValue;
  p.x = x;
  p.w = w;
  p.y = y;
  p.M = M;
  p.row0 = row0;
  return launch_rows<false>(p, pow2_at_least(M), s);
}

cudaError_t launch_stq1_mm_id(const float* x, const uint8_t* w, const int32_t* ids, float* y, int T, int N,
                              int K, int E, int* flags, cudaStream_t s) {
  Params p = base_params(N, K);
  p.x = x;
  p.w = w;
  p.y = y;
  p.ids = ids;
  p.flags = flags;
  p.T = T;
  p.E = E;
  p.flat = E <= 1024 ? 1 : 0;
  // Tokens per pass: twice the mean per expert (at least two), at most T and
  // the staging limit; an expert with more tokens takes more passes.
  long long want = 2LL * ((T + E - 1) / E);
  if (want < 2) want = 2;
  if (want > T) want = T;
  int R = pow2_at_least((int)want);
  if (R > p.xcap) R = p.xcap;
  p.xcap = R;
  return launch_rows<true>(p, R, s);
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

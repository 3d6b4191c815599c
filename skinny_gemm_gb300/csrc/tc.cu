// tc.cu -- tensor-core W4A16 skinny GEMM for sm_103a (activation rows eight at a time).
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
//   and y = bf16(((p_0 + p_1) + p_2) + ...).  A K that is not a multiple of
//   512 runs as K' = 512 ceil(K / 512): the padding groups read zero codes,
//   scales and biases (the out-of-bounds fill of the tensor copies) and zero
//   activations, so both of their fma steps add +0 to p_s.  Every kernel in this file
//   reproduces exactly this sequence, so row m of any call equals the M = 1
//   call bit for bit ([G4MK "Implementation notes": the verify GEMM is kept
//   arithmetic-identical to the sequential GEMV), and w4a16_mm_id rows equal
//   w4a16_mm on the selected expert.  An MMA output column depends only on
//   its own activation column, so unused columns (M < 8) change nothing.
//
// Data path of one warp:
//  * Packed codes stream HBM -> shared memory by TMA (cp.async.bulk.tensor,
//    128-byte swizzle), 32 rows x 512 codes (two 128-byte boxes, 8 KB) and
//    the 8 groups' scales and biases per stage, into a ring of `stages`
//    slots, each guarded by an mbarrier.  The stage's activation chunk (up
//    to 8 rows x 512 bf16) arrives by cp.async.bulk into padded rows of the
//    same slot, or the activation rows are staged once per CTA.  Lane 0
//    issues the copies; the ring runs ahead across work units, so DRAM
//    latency is paid once per warp, not once per tile.
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
// Launch shapes (the arithmetic above in every one):
//  * tc_tile_kernel -- shapes whose slices are single stages: a CTA (or a
//    cluster of CTAs splitting K) holds a 16- or 32-row tile's weights in
//    shared memory and adds the slice sums in slice order through
//    distributed shared memory; activation rows stream through eight at a
//    time.  Also w4a16_mm_group (several matrices in one grid) and, for
//    more than 32 tokens, w4a16_mm_id (one CTA per row tile and expert).
//  * tc_stream_kernel -- larger shapes: a persistent grid whose warps take
//    work units (32 rows x one K-slice) from a counter; with ksplit > 1 a
//    unit writes its fp32 partial to a workspace and bumps a per-tile
//    counter, and the warp that completes a tile adds the partials in slice
//    order (the result does not depend on which warp arrives last).  Its
//    routed mode serves w4a16_mm_id up to 32 tokens (whole-K units of the
//    chunks the ids select) and its argmax mode w4a16_mm_argmax.
//  * tc_routed_kernel -- w4a16_mm_id with the persistent shape selected and
//    more than 32 tokens: one CTA per (row tile, expert).
//
// No spin-wait is unbounded: an mbarrier wait that exceeds its iteration
// limit raises W4A16_DEVICE_TIMEOUT and the warp stops computing.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <map>
#include <mutex>
#include <set>
#include <utility>

#include "common.cuh"
#include "launch.h"
#include "route.cuh"

namespace w4a16 {
namespace {

// Tuning knobs (compile-time; the defaults are the measured choice).
#ifndef W4A16_TC_STREAM_WARPS
#define W4A16_TC_STREAM_WARPS 4    // warps per CTA of the persistent kernel (32-row warps)
#endif
#ifndef W4A16_TC_MIN_BLOCKS
#define W4A16_TC_MIN_BLOCKS 2      // persistent CTAs per SM the register budget must allow
#endif
#ifndef W4A16_TC_MAX_STAGES
#define W4A16_TC_MAX_STAGES 4      // deepest per-warp ring
#endif
#ifndef W4A16_TC_SMEM_TARGET
#define W4A16_TC_SMEM_TARGET (76 * 1024)  // shared memory per CTA the ring depth aims below
#endif
#ifndef W4A16_TC_GROUP_BATCH
#define W4A16_TC_GROUP_BATCH 2     // 64-groups whose loads and MMA chains are interleaved
#endif
#ifndef W4A16_TC_TILE_MAX_UNITS
// largest stages x 32-row tiles the tile kernel takes (measured: at 6144 units
// the tile kernel is 5-20% faster than the persistent grid, e.g. 24576x4096
// at M = 4 19.2 against 24.5 us; from 7168 units on it is slower)
#define W4A16_TC_TILE_MAX_UNITS 6655
#endif
#ifndef W4A16_TC_DYN_ALL
#define W4A16_TC_DYN_ALL 1  // 0: deal units round-robin when K is not split
#endif
#ifndef W4A16_TC_STREAM_NSUB1_MIN_M
#define W4A16_TC_STREAM_NSUB1_MIN_M 9  // smallest chunk the persistent kernel runs with 16-row warps
#endif
#ifndef W4A16_TC_TILE_SLICES_PER_WARP
#define W4A16_TC_TILE_SLICES_PER_WARP 1  // K-slices one warp of the tile kernel computes (in turn)
#endif
#ifndef W4A16_TC_TILE_SLICES
#define W4A16_TC_TILE_SLICES 5        // most K-slices one CTA of the tile kernel takes, where a cluster can split
#endif
#ifndef W4A16_TC_PIPE
#define W4A16_TC_PIPE 1  // persistent kernel: software-pipelined stage computation
#endif
#ifndef W4A16_TC_PIPE_BATCH
#define W4A16_TC_PIPE_BATCH 1  // 64-groups per batch of the pipelined stage
#endif

constexpr int kTileRows = 32;           // two m16 subtiles per warp
constexpr int kBoxWords = 32;           // one TMA box row: 128 bytes = 256 codes
constexpr int kBoxBytes = kTileRows * kBoxWords * 4;            // 4096
constexpr int kStageK = 512;            // codes per stage per row (two boxes)
constexpr int kStageWords = kStageK / 8;
constexpr int kCodeBytes = 2 * kBoxBytes;                        // 8192 codes per stage
constexpr int kParamBytes = kTileRows * 8 * 2;                   // 512: 8 bf16 per row per stage
constexpr int kCodeSlotBytes = kCodeBytes + 2 * kParamBytes;     // 9216: codes | scales | biases
constexpr int kXPitch = kStageK * 2 + 64;                        // 1088: conflict-free LDS.128

// K rounded up to whole stages (the logical K of the canonical arithmetic).
__host__ __device__ constexpr int kpad(int K) { return (K + kStageK - 1) / kStageK * kStageK; }
constexpr int kRoutedWarps = 8;          // max warps per CTA of the routed kernel
#ifndef W4A16_TC_TARGET_UNITS
#define W4A16_TC_TARGET_UNITS (152 * 16)
#endif
constexpr int kTargetUnits = W4A16_TC_TARGET_UNITS;  // work units wanted per chunk (~16 per SM)
constexpr int kSmemLimit = 227 * 1024;
constexpr uint32_t kWaitLimit = 1u << 20;
constexpr uint32_t kMagic = 0x43004300u;  // two bf16 128.0
constexpr uint32_t kOnes = 0x3F803F80u;   // two bf16 1.0

// Geometry of a work unit of 16 * NSUB rows (NSUB m16 subtiles per warp):
// one 128-byte TMA box row per row, two boxes (512 codes) per stage, then
// the stage's 8 scales and 8 biases per row; slots are kept 1 KB aligned
// for the 128-byte swizzle.
template <int NSUB>
struct Geo {
  static constexpr int kRows = 16 * NSUB;
  static constexpr int kBox = kRows * 128;
  static constexpr int kParam = kRows * 16;
  static constexpr int kSlot = (2 * kBox + 2 * kParam + 1023) / 1024 * 1024;  // 9216 | 5120
  static constexpr int kCodeSlot = (2 * kBox + 1023) / 1024 * 1024;            // codes only: 8192 | 4096
  static constexpr int kWarps = NSUB == 2 ? W4A16_TC_STREAM_WARPS : 8;  // warps per CTA of the persistent kernel
};

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

// Bounded wait: true when the phase completed, false after `limit` tries.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t limit = kWaitLimit) {
  for (uint32_t i = 0; i < limit; ++i)
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

// L2 eviction policies: the packed codes are read exactly once and go first;
// activations and group parameters are reused and should stay.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int cx, int cy, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(dst), "l"(map), "r"(cx), "r"(cy), "r"(bar), "l"(policy)
      : "memory");
}

// A box of the tensor into L2 only (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2(const CUtensorMap* map, int cx, int cy) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(cx), "r"(cy)
               : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Programmatic dependent launch.  launch_dependents lets the next kernel on
// the stream start its CTAs (and their prologue) while this one runs; wait
// blocks until every kernel this one depends on has completed and its writes
// are visible.  Without a programmatic dependency both are no-ops.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Relaxed load at GPU scope (a counter other CTAs update atomically).
// Release / acquire fence at GPU scope: with a relaxed atomic after (before)
// it, the partial sums stored before it are visible to the warp that sees
// the count.  Lighter than the sequentially consistent fence.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ int ld_relaxed_gpu(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

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


__device__ __forceinline__ float half_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float half_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// ---- one warp's stage ring -------------------------------------------------------------

struct Ring {
  uint32_t codes0, xs0, bars0;
  int S, x_slot;
  uint32_t issued, consumed;
  uint64_t pol_stream, pol_keep;
  uint32_t limit = kWaitLimit;  // tries of a stage wait before the warp gives up
};

// Lane 0 only: start the loads of stage `st` (codes of 32 rows from
// tensor_row: two 128-byte boxes; x of the listed activation rows) into the
// next free slot.
struct Maps {
  CUtensorMap codes;   // u32 [rows][K/8], box 32 words x 32 rows, 128-byte swizzle
  CUtensorMap scales;  // bf16 [rows][K/64], box 8 groups x 32 rows
  CUtensorMap biases;
};

// The weight part of a stage: codes (two boxes, to dst) and the 8 groups'
// scales and biases (to pdst) of 16 * NSUB rows from tensor_row; arms `bar`
// for those bytes plus `mc` activation chunks still to come.
// With PARAMS false only the codes are requested (group-128 tables and
// K % 512 != 0 bring their parameters per work unit instead).  box1 false:
// the stage's second box lies wholly past K (the last stage of a padded K)
// and is not requested; its slot keeps older codes, which meet zero
// activations and zero parameters there.
template <int NSUB, bool PARAMS = true>
__device__ __forceinline__ void issue_weights(uint32_t dst, uint32_t pdst, uint32_t bar, const Maps* maps, int st,
                                              int tensor_row, int mc, uint64_t pol_stream, uint64_t pol_keep,
                                              uint32_t extra_bytes = 0, bool box1 = true) {
  using G = Geo<NSUB>;
  mbar_expect_tx(bar, (box1 ? 2 : 1) * G::kBox + (PARAMS ? 2 * G::kParam : 0) + (uint32_t)(mc * kStageK * 2) +
                          extra_bytes);
  tma_load_2d(dst, &maps->codes, st * kStageWords, tensor_row, bar, pol_stream);
  if (box1) tma_load_2d(dst + G::kBox, &maps->codes, st * kStageWords + kBoxWords, tensor_row, bar, pol_stream);
  if (PARAMS) {
    tma_load_2d(pdst, &maps->scales, st * 8, tensor_row, bar, pol_keep);
    tma_load_2d(pdst + G::kParam, &maps->biases, st * 8, tensor_row, bar, pol_keep);
  }
}

// Zeros for the activation padding past K (at most 448 bf16 of a row).
__device__ __align__(128) uint4 g_xzero[64] = {};

// The activation part of a stage: 512 bf16 of each row toks[0..mc) into rows
// of kXPitch bytes at xdst; in the last stage of a K % 512 != 0 shape the
// codes past K are zeros (a second copy, so the stage's byte count is the same).
__device__ __forceinline__ void issue_x(uint32_t xdst, uint32_t bar, int st, const uint16_t* x, const int* toks,
                                        int mc, int K, uint64_t pol_keep) {
  const uint16_t* xs = x + (int64_t)st * kStageK;
  const int valid = min(kStageK, K - st * kStageK);  // a multiple of 64
  for (int n = 0; n < mc; ++n) {
    bulk_load(xdst + n * kXPitch, xs + (int64_t)toks[n] * K, valid * 2, bar, pol_keep);
    if (valid < kStageK) bulk_load(xdst + n * kXPitch + valid * 2, g_xzero, (kStageK - valid) * 2, bar, pol_keep);
  }
}

// Lane 0 only: the weights of stage `st` into the next free slot; returns the
// slot.  `extra` bytes are expected on top of what the copies deliver (the
// debug fault that lets a stage wait run out; 0 otherwise).
template <int NSUB>
__device__ __forceinline__ uint32_t ring_issue_w(Ring& R, const Maps* maps, int st, int tensor_row, int mc,
                                                 uint32_t extra = 0) {
  const uint32_t slot = R.issued % (uint32_t)R.S;
  const uint32_t dst = R.codes0 + slot * Geo<NSUB>::kSlot;
  issue_weights<NSUB>(dst, dst + 2 * Geo<NSUB>::kBox, R.bars0 + 8 * slot, maps, st, tensor_row, mc, R.pol_stream,
                      R.pol_keep, extra);
  ++R.issued;
  return slot;
}

// Lane 0 only: the activation chunks of stage `st` into `slot`.
__device__ __forceinline__ void ring_issue_x(const Ring& R, uint32_t slot, int st, const uint16_t* x, const int* toks,
                                             int mc, int K) {
  issue_x(R.xs0 + slot * R.x_slot, R.bars0 + 8 * slot, st, x, toks, mc, K, R.pol_keep);
}

template <int NSUB>
__device__ __forceinline__ void ring_issue(Ring& R, const Maps* maps, int st, int tensor_row, const uint16_t* x,
                                           const int* toks, int mc, int K) {
  const uint32_t slot = ring_issue_w<NSUB>(R, maps, st, tensor_row, mc);
  ring_issue_x(R, slot, st, x, toks, mc, K);
}

// All lanes: wait for the oldest outstanding slot.  Returns false on timeout.
__device__ __forceinline__ bool ring_wait(Ring& R, uint32_t& slot) {
  slot = R.consumed % (uint32_t)R.S;
  const uint32_t parity = (R.consumed / (uint32_t)R.S) & 1u;
  const bool ok = mbar_wait(R.bars0 + 8 * slot, parity, R.limit);
  return __all_sync(0xffffffffu, ok);
}

// Activation B fragments of one 16-byte chunk x0..x7 of a column: for the
// code pairing (i, i+4) of a packed word, h = 0 takes (x0,x4),(x1,x5) and
// h = 1 takes (x2,x6),(x3,x7).
__device__ __forceinline__ void frag_from_chunk(const uint4& u, uint32_t (&b)[2][2]) {
  b[0][0] = prmt(u.x, u.z, 0x5410);
  b[0][1] = prmt(u.x, u.z, 0x7632);
  b[1][0] = prmt(u.y, u.w, 0x5410);
  b[1][1] = prmt(u.y, u.w, 0x7632);
}

__device__ __forceinline__ float2 lds64f(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint32_t component(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Per-lane byte offsets of the ldmatrix rows inside a 128-byte-swizzled box,
// for subtile s and group-in-box gl: rows g / g+8, chunks 2gl and 2gl+1.
__device__ __forceinline__ void ldsm_offsets(int lane, uint32_t (&off)[2][4]) {
  const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int gl = 0; gl < 4; ++gl) {
      const int row = 16 * s + 8 * (mi & 1) + r8;
      const int chunk = 2 * gl + (mi >> 1);
      off[s][gl] = (uint32_t)(row * 128 + ((chunk ^ r8) << 4));
    }
}

// One stage (16 NSUB rows x 512 codes, 8 groups) of the canonical recurrence
// into p[s][i]: subtile s, i = (row g: columns 2t, 2t+1; row g+8: columns 2t,
// 2t+1).  GB groups at a time: their loads are issued first and their MMA
// chains interleaved.  With ALLCOLS false (one activation row) the odd
// columns are not rescaled; the even columns' arithmetic is unchanged.
__device__ __forceinline__ uint2 lds64u(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds32u(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds16u(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// 16 bytes at a shared address aligned to `al` bytes (2, 4 or 8; warp-uniform).
__device__ __forceinline__ uint4 lds128_al(uint32_t a, uint32_t al) {
  if (al >= 8) {
    const uint2 lo = lds64u(a), hi = lds64u(a + 8);
    return make_uint4(lo.x, lo.y, hi.x, hi.y);
  }
  if (al == 4) return make_uint4(lds32u(a), lds32u(a + 4), lds32u(a + 8), lds32u(a + 12));
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) w[k] = lds16u(a + 4 * k) | (lds16u(a + 4 * k + 2) << 16);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Where the stage's scales and biases are read (PM):
//  0: the stage's own boxes, 16 bytes per row, BOXROWS rows of scales then of
//     biases at pbase (pbase pointing at the warp's first row);
//  1 (G128): a table with one scale and bias per 128 codes (the stage's 8
//     64-groups use 4 of each), read at pbase + r * prow (scales) and
//     pbase + pbias + r * prow (biases), 8 bytes per row.  Each 64-group is
//     rescaled with its 128-group's pair: the arithmetic of the group-64
//     kernel on a table whose pairs repeat over the two halves of every
//     128-group;
//  2 (K % 512 != 0): a work unit's group-64 rows as they lie in memory, K / 32
//     bytes apart: 16 bytes at pbase + r * prow (and + pbias), aligned to
//     `pal` bytes; in the last stage the groups from `gv` on lie past K (the
//     bytes there are the next row's) and read as zero.
template <int NSUB, int BOXROWS, int PM>
__device__ __forceinline__ void stage_params(uint4 (&ps)[2 * NSUB], uint4 (&pb)[2 * NSUB], uint32_t pbase, int g,
                                             uint32_t prow, uint32_t pbias, uint32_t pal, int gv) {
  constexpr uint32_t kBiases = BOXROWS * 16;
#pragma unroll
  for (int i = 0; i < 2 * NSUB; ++i) {
    const uint32_t r = 16 * (i >> 1) + g + 8 * (i & 1);
    if (PM == 1) {
      const uint2 s2 = lds64u(pbase + r * prow), b2 = lds64u(pbase + pbias + r * prow);
      ps[i] = make_uint4(s2.x, s2.y, 0u, 0u);
      pb[i] = make_uint4(b2.x, b2.y, 0u, 0u);
    } else if (PM == 2) {
      ps[i] = lds128_al(pbase + r * prow, pal);
      pb[i] = lds128_al(pbase + pbias + r * prow, pal);
    } else {
      ps[i] = lds128(pbase + r * 16);
      pb[i] = lds128(pbase + kBiases + r * 16);
    }
  }
  if (PM == 2 && gv < 8) {
    uint32_t mk[4];  // word w holds groups 2w (low half) and 2w + 1
#pragma unroll
    for (int w = 0; w < 4; ++w) mk[w] = 2 * w + 1 < gv ? 0xFFFFFFFFu : 2 * w < gv ? 0x0000FFFFu : 0u;
#pragma unroll
    for (int i = 0; i < 2 * NSUB; ++i) {
      ps[i] = make_uint4(ps[i].x & mk[0], ps[i].y & mk[1], ps[i].z & mk[2], ps[i].w & mk[3]);
      pb[i] = make_uint4(pb[i].x & mk[0], pb[i].y & mk[1], pb[i].z & mk[2], pb[i].w & mk[3]);
    }
  }
}

template <int NSUB, bool ALLCOLS, bool XSTAGED, int BOXROWS = 16 * NSUB, int PM = 0>
__device__ __forceinline__ void compute_stage(uint32_t cbase, uint32_t pbase, uint32_t xbase, bool xvalid,
                                              uint32_t sxbase, uint32_t sx_stride, bool xvalid_cols,
                                              float (&p)[NSUB][4], const uint32_t (&loff)[NSUB][4], int g,
                                              uint32_t prow = 0, uint32_t pbias = 0, uint32_t pal = 16,
                                              int gv = 8) {
  constexpr int GB = W4A16_TC_GROUP_BATCH;
  constexpr bool G128 = PM == 1;
  // Codes: two boxes of BOXROWS rows x 128 bytes at cbase (the warp's rows
  // picked by loff); the parameters as stage_params reads them.
  constexpr uint32_t kBox = BOXROWS * 128;
  // scale / bias of the 8 groups for this lane's rows 16(i>>1) + g + 8(i&1)
  uint4 ps[2 * NSUB], pb[2 * NSUB];
  stage_params<NSUB, BOXROWS, PM>(ps, pb, pbase, g, prow, pbias, pal, gv);
#pragma unroll
  for (int gp = 0; gp < 8; gp += GB) {
    uint32_t w[GB][NSUB][4];  // [group][subtile]: rows g / g+8 of chunk 2gl, then of chunk 2gl+1
    uint4 u[GB][2];           // [group][chunk] activations
#pragma unroll
    for (int j = 0; j < GB; ++j) {
      const int gi = gp + j;
#pragma unroll
      for (int s = 0; s < NSUB; ++s)
        ldsm_x4(cbase + (gi >> 2) * kBox + loff[s][gi & 3], w[j][s][0], w[j][s][1], w[j][s][2], w[j][s][3]);
#pragma unroll
    for (int cb = 0; cb < 2; ++cb) {
        u[j][cb] = make_uint4(0, 0, 0, 0);
        if (xvalid) u[j][cb] = lds128(xbase + 128 * gi + 64 * cb);
      }
    }
    uint32_t bx[GB][2][2][2];  // [group][chunk][h][reg]
    float sx[GB][4], acc[GB][NSUB][4];
#pragma unroll
    for (int j = 0; j < GB; ++j) {
#pragma unroll
      for (int cb = 0; cb < 2; ++cb) {
        if (XSTAGED) {  // already in fragment order
          bx[j][cb][0][0] = u[j][cb].x;
          bx[j][cb][0][1] = u[j][cb].y;
          bx[j][cb][1][0] = u[j][cb].z;
          bx[j][cb][1][1] = u[j][cb].w;
        } else {
          frag_from_chunk(u[j][cb], bx[j][cb]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sx[j][i] = 0.f;
#pragma unroll
        for (int s = 0; s < NSUB; ++s) acc[j][s][i] = 0.f;
      }
      if (XSTAGED && xvalid_cols) {  // precomputed group sums of columns 2t, 2t+1
        const float2 v = lds64f(sxbase + sx_stride * (gp + j));
        sx[j][0] = v.x;
        sx[j][1] = v.y;
      }
    }
    // the four (chunk, h) steps of every chain, in the canonical order, chains interleaved
#pragma unroll
    for (int step = 0; step < 4; ++step) {
      const int cb = step >> 1, h = step & 1;
#pragma unroll
      for (int j = 0; j < GB; ++j) {
        if (!XSTAGED) mma_bf16(sx[j], kOnes, kOnes, kOnes, kOnes, bx[j][cb][h][0], bx[j][cb][h][1]);
#pragma unroll
        for (int s = 0; s < NSUB; ++s) {
          const uint32_t wg = w[j][s][2 * cb], wg8 = w[j][s][2 * cb + 1];
          const uint32_t a0 = codes_as_bf16x2(wg >> (8 * h));
          const uint32_t a1 = codes_as_bf16x2(wg8 >> (8 * h));
          const uint32_t a2 = codes_as_bf16x2(wg >> (8 * h + 4));
          const uint32_t a3 = codes_as_bf16x2(wg8 >> (8 * h + 4));
          mma_bf16(acc[j][s], a0, a1, a2, a3, bx[j][cb][h][0], bx[j][cb][h][1]);
        }
      }
    }
    // group rescale, groups in order
#pragma unroll
    for (int j = 0; j < GB; ++j) {
      const int gi = gp + j;
#pragma unroll
      for (int s = 0; s < NSUB; ++s)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const int i = 2 * s + rr;
          const int pi = G128 ? gi >> 1 : gi;  // this group's parameter pair in the row's stage slice
          const uint32_t sw = component(ps[i], pi >> 1);
          const uint32_t bw = component(pb[i], pi >> 1);
          const float sc = (pi & 1) ? half_hi(sw) : half_lo(sw);
          const float bi = (pi & 1) ? half_hi(bw) : half_lo(bw);
          const float cc = __fmaf_rn(-128.0f, sc, bi);
          p[s][2 * rr + 0] = __fmaf_rn(sc, acc[j][s][2 * rr + 0], p[s][2 * rr + 0]);
          p[s][2 * rr + 0] = __fmaf_rn(cc, sx[j][0], p[s][2 * rr + 0]);
          if (ALLCOLS) {
            p[s][2 * rr + 1] = __fmaf_rn(sc, acc[j][s][2 * rr + 1], p[s][2 * rr + 1]);
            p[s][2 * rr + 1] = __fmaf_rn(cc, sx[j][1], p[s][2 * rr + 1]);
          }
        }
    }
  }
}

// The same stage, software-pipelined for a warp that has the registers: the
// shared-memory loads of group batch b + 1 go out before the MMAs of batch
// b, and the rescale of batch b waits until the MMAs of batch b + 1 are
// issued (its accumulators are complete by then).  Every p receives the
// same operations in the same order as compute_stage, so the bits agree.
template <int NSUB, bool ALLCOLS, bool XSTAGED, int BOXROWS = 16 * NSUB, int PM = 0>
__device__ __forceinline__ void compute_stage_pipe(uint32_t cbase, uint32_t pbase, uint32_t xbase, bool xvalid,
                                                   uint32_t sxbase, uint32_t sx_stride, bool xvalid_cols,
                                                   float (&p)[NSUB][4], const uint32_t (&loff)[NSUB][4], int g,
                                                   uint32_t prow = 0, uint32_t pbias = 0, uint32_t pal = 16,
                                                   int gv = 8) {
  constexpr int GB = W4A16_TC_PIPE_BATCH, NB = 8 / GB;
  constexpr bool G128 = PM == 1;
  constexpr uint32_t kBox = BOXROWS * 128;
  uint4 ps[2 * NSUB], pb[2 * NSUB];
  stage_params<NSUB, BOXROWS, PM>(ps, pb, pbase, g, prow, pbias, pal, gv);
  // Batch b uses buffer b % 2 of the loads and accumulators and b % 3 of the
  // group sums: those of batch b - 1 are still to be read by its rescale
  // when batch b + 1 is loaded.
  uint32_t w[2][GB][NSUB][4];   // [buffer][group][subtile] code words
  uint4 u[2][GB][2];            // [buffer][group][chunk] activations
  float sx[3][GB][4];           // [buffer][group] group sums
  float acc[2][GB][NSUB][4];    // [buffer][group][subtile]
  auto load = [&](int b, int buf) {
    const int sb = b % 3;
#pragma unroll
    for (int j = 0; j < GB; ++j) {
      const int gi = b * GB + j;
#pragma unroll
      for (int s = 0; s < NSUB; ++s)
        ldsm_x4(cbase + (gi >> 2) * kBox + loff[s][gi & 3], w[buf][j][s][0], w[buf][j][s][1], w[buf][j][s][2],
                w[buf][j][s][3]);
#pragma unroll
      for (int cb = 0; cb < 2; ++cb) {
        u[buf][j][cb] = make_uint4(0, 0, 0, 0);
        if (xvalid) u[buf][j][cb] = lds128(xbase + 128 * gi + 64 * cb);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) sx[sb][j][i] = 0.f;
      if (XSTAGED && xvalid_cols) {
        const float2 v = lds64f(sxbase + sx_stride * gi);
        sx[sb][j][0] = v.x;
        sx[sb][j][1] = v.y;
      }
    }
  };
  auto mmas = [&](int b, int buf) {
    const int sb = b % 3;
    uint32_t bx[GB][2][2][2];
#pragma unroll
    for (int j = 0; j < GB; ++j) {
#pragma unroll
      for (int cb = 0; cb < 2; ++cb) {
        if (XSTAGED) {
          bx[j][cb][0][0] = u[buf][j][cb].x;
          bx[j][cb][0][1] = u[buf][j][cb].y;
          bx[j][cb][1][0] = u[buf][j][cb].z;
          bx[j][cb][1][1] = u[buf][j][cb].w;
        } else {
          frag_from_chunk(u[buf][j][cb], bx[j][cb]);
        }
      }
#pragma unroll
      for (int s = 0; s < NSUB; ++s)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[buf][j][s][i] = 0.f;
    }
#pragma unroll
    for (int step = 0; step < 4; ++step) {
      const int cb = step >> 1, h = step & 1;
#pragma unroll
      for (int j = 0; j < GB; ++j) {
        if (!XSTAGED) mma_bf16(sx[sb][j], kOnes, kOnes, kOnes, kOnes, bx[j][cb][h][0], bx[j][cb][h][1]);
#pragma unroll
        for (int s = 0; s < NSUB; ++s) {
          const uint32_t wg = w[buf][j][s][2 * cb], wg8 = w[buf][j][s][2 * cb + 1];
          const uint32_t a0 = codes_as_bf16x2(wg >> (8 * h));
          const uint32_t a1 = codes_as_bf16x2(wg8 >> (8 * h));
          const uint32_t a2 = codes_as_bf16x2(wg >> (8 * h + 4));
          const uint32_t a3 = codes_as_bf16x2(wg8 >> (8 * h + 4));
          mma_bf16(acc[buf][j][s], a0, a1, a2, a3, bx[j][cb][h][0], bx[j][cb][h][1]);
        }
      }
    }
  };
  auto rescale = [&](int b, int buf) {
    const int sb = b % 3;
#pragma unroll
    for (int j = 0; j < GB; ++j) {
      const int gi = b * GB + j;
#pragma unroll
      for (int s = 0; s < NSUB; ++s)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const int i = 2 * s + rr;
          const int pi = G128 ? gi >> 1 : gi;
          const uint32_t sw = component(ps[i], pi >> 1);
          const uint32_t bw = component(pb[i], pi >> 1);
          const float sc = (pi & 1) ? half_hi(sw) : half_lo(sw);
          const float bi = (pi & 1) ? half_hi(bw) : half_lo(bw);
          const float cc = __fmaf_rn(-128.0f, sc, bi);
          p[s][2 * rr + 0] = __fmaf_rn(sc, acc[buf][j][s][2 * rr + 0], p[s][2 * rr + 0]);
          p[s][2 * rr + 0] = __fmaf_rn(cc, sx[sb][j][0], p[s][2 * rr + 0]);
          if (ALLCOLS) {
            p[s][2 * rr + 1] = __fmaf_rn(sc, acc[buf][j][s][2 * rr + 1], p[s][2 * rr + 1]);
            p[s][2 * rr + 1] = __fmaf_rn(cc, sx[sb][j][1], p[s][2 * rr + 1]);
          }
        }
    }
  };
  load(0, 0);
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    if (b + 1 < NB) load(b + 1, (b + 1) & 1);
    mmas(b, b & 1);
    if (b > 0) rescale(b - 1, (b - 1) & 1);
  }
  rescale(NB - 1, (NB - 1) & 1);
}

// The persistent kernel's stage: pipelined unless W4A16_TC_PIPE is 0.
template <int NSUB, bool ALLCOLS, bool XSTAGED, int BOXROWS = 16 * NSUB, int PM = 0>
__device__ __forceinline__ void compute_stage_sel(uint32_t cbase, uint32_t pbase, uint32_t xbase, bool xvalid,
                                                  uint32_t sxbase, uint32_t sx_stride, bool xvalid_cols,
                                                  float (&p)[NSUB][4], const uint32_t (&loff)[NSUB][4], int g,
                                                  uint32_t prow = 0, uint32_t pbias = 0, uint32_t pal = 16,
                                                  int gv = 8) {
#if W4A16_TC_PIPE
  compute_stage_pipe<NSUB, ALLCOLS, XSTAGED, BOXROWS, PM>(cbase, pbase, xbase, xvalid, sxbase, sx_stride,
                                                          xvalid_cols, p, loff, g, prow, pbias, pal, gv);
#else
  compute_stage<NSUB, ALLCOLS, XSTAGED, BOXROWS, PM>(cbase, pbase, xbase, xvalid, sxbase, sx_stride, xvalid_cols,
                                                     p, loff, g, prow, pbias, pal, gv);
#endif
}

struct Shape {
  int nst, tiles, sl, ks, units;
};

__host__ __device__ inline Shape tc_shape(int N, int K) {
  Shape s;
  s.nst = kpad(K) / kStageK;
  s.tiles = (N + kTileRows - 1) / kTileRows;
  int64_t sl = (int64_t)s.nst * s.tiles / kTargetUnits;
  if (sl < 1) sl = 1;
  if (sl > s.nst) sl = s.nst;
  s.sl = (int)sl;
  s.ks = (s.nst + s.sl - 1) / s.sl;
  s.units = s.tiles * s.ks;
  return s;
}

// codes_only: stage slots without the parameter boxes (the parameters come
// per work unit instead, K % 512 != 0)
template <int NSUB>
__host__ __device__ inline int ring_bytes(int stages, int mcap, bool codes_only = false) {
  return stages * ((codes_only ? Geo<NSUB>::kCodeSlot : Geo<NSUB>::kSlot) + mcap * kXPitch);
}

// ---- persistent kernel (w4a16_mm) ------------------------------------------------------

// Bytes after the barriers: token rows [8] and every warp's unit ring [8] (ints).
// tokens [8] | dealt units [8 warps][8] | activation barrier
constexpr int kStreamMisc = 4 * (kMaxChunk + 8 * 8) + 32;
// argmax mode, after the pre-staged activations: best keys [8 warps][8
// columns] and the CTA's [8] (u64)
constexpr int kArgmaxSmem = 8 * (8 * 8 + 8);

struct StreamParams {
  const uint16_t* x;
  const uint16_t* S;
  const uint16_t* B;
  uint16_t* y;
  float* part;      // [units][8][rows] slice partials (ksplit > 1)
  int* cnt;         // [tiles] arrival counters, zero between launches
  int* sched;       // [1] unit-grab counter, zero between launches
  int* flags;
  int N, K, M, row0;
  int nst, sl, ks, tiles, units;  // tiles and units of 16 * NSUB rows
  int kfull;        // slices of full length per tile: ks, or ks - 1 when the last is shorter
  int stages;
  int xpitch;       // bytes per activation row of the pre-staged copy (0: per-stage copies)
  int prefetch;     // request the first weight stages before waiting for earlier kernels
  int g128;         // scales and biases are [N][K/128] (one pair per 128 codes)
  int ptail;        // K % 512 != 0: whole-K units, each with its parameter rows by bulk copy
  int fault_tx;     // debug: bytes the first stage of CTA 0's warp 0 expects beyond its copies
  uint32_t wait_limit;  // tries of a stage wait (0: the default)
  int l2_stages;        // routed mode: leading stages of every expert pulled into L2 before the ids are known
  int par_off;      // g128 / ptail: byte offset of the per-unit parameter slots in shared memory
  const int32_t* ids;  // routed mode: expert id of each of T tokens, E experts of N rows each
  int T, E;
  unsigned long long* best;  // argmax mode: [8] running keys, zero between launches
  int* done;                 // and the finished-CTA counter, zero between launches
  int32_t* idx;              // argmax of activation row row0 + n over the N outputs
  uint16_t* val;             // and its value (may be null)
};

// Argmax mode: an output value as a key whose unsigned order is the value's
// order (bf16 bits mapped to an order-preserving 16-bit code, every NaN
// above +inf), ties going to the smaller row n.
__device__ __forceinline__ unsigned long long argmax_key(uint16_t b, int n) {
  const bool nan = (b & 0x7F80u) == 0x7F80u && (b & 0x7Fu) != 0u;
  const uint32_t ord = nan ? 0xFFFFu : (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
  return ((unsigned long long)ord << 32) | (0xFFFFFFFFu - (uint32_t)n);
}

__device__ __forceinline__ unsigned long long max_u64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}

// Maximum over the lanes given by the xor masks from `from` down to 1.
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long k, int from, int to) {
  for (int m = from; m >= to; m >>= 1) k = max_u64(k, __shfl_xor_sync(0xffffffffu, k, m));
  return k;
}

// Tile and slice of work unit u.  Units whose slice has the full length come
// first, tile-major; the shorter last slice of every tile (when the slice
// length does not divide the stage count) comes after all of them, so the
// units dealt last are the shortest and the warps finish closer together.
// The order of the units changes no result: every partial has its fixed
// place and the sums run in slice order.
template <bool SPLIT>
__device__ __forceinline__ int unit_tile(const StreamParams& p, int u, int& slice) {
  if (!SPLIT) {
    slice = 0;
    return u;
  }
  const int nfull = p.tiles * p.kfull;
  if (u >= nfull) {
    slice = p.ks - 1;
    return u - nfull;
  }
  const int tile = u / p.kfull;  // one division per unit
  slice = u - tile * p.kfull;
  return tile;
}

// Columns of the group-sum table: the even count >= mc (lane t reads columns 2t, 2t+1).
__host__ __device__ inline int sx_cols(int mc) { return (mc + 1) & ~1; }

// Bytes of shared memory the pre-staged activations and their group sums
// take: mc rows of 2K + 64 bytes (fragment order, padded for conflict-free
// reads) and K/64 groups x sx_cols(mc) fp32 sums; K here is the padded kpad(K).
__host__ __device__ inline int xstage_bytes(int mc, int K) {
  return mc * (2 * K + 64) + (K / kGroup) * sx_cols(mc) * 4;
}

// Persistent CTAs of Geo<NSUB>::kWarps warps; a warp's work unit is
// 16 * NSUB rows x one K-slice.  With NSUB = 1 a warp needs half the
// registers and shared memory, so twice as many warps fit on an SM.
template <int NSUB>
constexpr int stream_min_blocks() { return NSUB == 1 ? 2 : Geo<NSUB>::kWarps >= 8 ? 1 : W4A16_TC_MIN_BLOCKS; }

// Routed mode: the chunk table every CTA builds from the expert ids after the
// wait for earlier kernels.  The tokens of each expert, in token order, form
// chunks of at most `cap` tokens; a chunk is one expert and its token rows.
// Chunks are numbered in the order of their first tokens (the order changes
// no result: every chunk writes its own rows with the canonical arithmetic).
// Layout (ints): [0] chunks, [1] tokens with an id out of range, then per
// chunk its expert, its token count and kMaxChunk tokens, then the
// out-of-range tokens.
constexpr int kRoutedStreamMaxT = 32;  // tokens the routed mode takes: one per lane
__host__ __device__ inline int routed_table_bytes(int T) { return (2 + T * (2 + kMaxChunk) + T) * 4; }

// Warp 0 only, T <= 32, token t in lane t.  Warp match and ballot only: no
// loop over tokens or experts.
__device__ __forceinline__ void build_chunks(const int32_t* __restrict__ ids, int T, int E, int cap, int* tab) {
  const int lane = threadIdx.x & 31;
  const int v = lane < T ? ids[lane] : -1;
  const bool ok = lane < T && v >= 0 && v < E;
  const int key = ok ? v : -1;
  const unsigned lt = (1u << lane) - 1u;
  const unsigned same = __match_any_sync(0xffffffffu, key);       // tokens of this expert
  const int before = __popc(same & lt);                            // ... ahead of this one
  const bool start = ok && before % cap == 0;                      // first token of a chunk
  // the tokens of this token's chunk (expert, chunk within the expert); its
  // lowest lane starts the chunk
  const unsigned mine = __match_any_sync(0xffffffffu, ok ? key * 32 + before / cap : -1);
  const unsigned starts = __ballot_sync(0xffffffffu, start);
  const int c = __popc(starts & ((1u << (__ffs(mine) - 1)) - 1u));  // chunks that start earlier
  if (ok) {
    int* ch = tab + 2 + c * (2 + kMaxChunk);
    ch[2 + before % cap] = lane;
    if (start) {
      ch[0] = key;
      ch[1] = min(cap, __popc(same) - before);
    }
  }
  const bool bad = lane < T && !ok;
  const unsigned badm = __ballot_sync(0xffffffffu, bad);
  if (bad) tab[2 + T * (2 + kMaxChunk) + __popc(badm & lt)] = lane;
  if (lane == 0) {
    tab[0] = __popc(starts);
    tab[1] = __popc(badm);
  }
}

// SPLIT: K is split over several units per tile (ks > 1).  The units after
// a warp's first are grabbed from a counter (LM head 262144x2560: 66.3 ->
// 65.3 us against round-robin dealing; 262144x1536 and 16384^2 unchanged).
// ROUTED (w4a16_mm_id): a unit is one chunk of tokens routed to one expert
// times one tile of that expert, over the whole K; the slice sums are folded
// in slice order as they complete, so every row equals w4a16_mm on the
// selected expert bit for bit.  Units are dealt round-robin over the chunks
// the ids select, so only the weights of experts with tokens are read.
// ARGMAX (w4a16_mm_argmax): the outputs are not stored; every warp keeps the
// largest key of each activation row over its units, the CTAs merge theirs
// with 64-bit atomic maxima, and the last CTA out writes the argmax of every
// row (the outputs' bits are those w4a16_mm stores).
template <int NSUB, bool ALLCOLS, bool XSTAGED, bool SPLIT, bool ROUTED = false, bool ARGMAX = false,
          bool WHOLEK = false, bool G128 = false, bool PT = false>
__global__ void __launch_bounds__(Geo<NSUB>::kWarps * 32, ROUTED ? 2 : stream_min_blocks<NSUB>()) tc_stream_kernel(
    const __grid_constant__ Maps maps, StreamParams p) {
  using G = Geo<NSUB>;
  constexpr int kW = G::kWarps, kRows = G::kRows;
  static_assert(!ROUTED || (!XSTAGED && !SPLIT), "the routed mode copies activations per stage, whole-K units");
  static_assert(!ARGMAX || (!ROUTED && NSUB == 2), "argmax over plain 32-row units");
  static_assert(!WHOLEK || (!ROUTED && !SPLIT && !ARGMAX), "whole-K units are a plain-mode schedule");
  static_assert(!G128 || (!ROUTED && !SPLIT && !ARGMAX), "group-128 tables: plain whole-K units");
  static_assert(!PT || (!ARGMAX && !G128), "K % 512 != 0: plain (whole-K or split) or routed units");
  constexpr bool DYN = (SPLIT || W4A16_TC_DYN_ALL) && !ROUTED;  // units after the first from the counter
  // whole-K units: slice sums folded in registers, in slice order
  constexpr bool FOLD = ROUTED || WHOLEK || G128 || (PT && !SPLIT);
  constexpr bool UBLK = G128 || PT;  // a unit's parameter rows come by bulk copy
  // Without a workspace (p.sched == nullptr) the units are dealt inside each
  // CTA: CTA c owns the contiguous units [c U / grid, (c + 1) U / grid) and
  // its warps take them from a shared-memory counter.  With one, from a
  // counter shared by the whole grid.
  const bool local = p.sched == nullptr;
  extern __shared__ uint8_t smem_raw[];
  pdl_launch_dependents();
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int S = p.stages, mc = p.M;   // routed mode: mc = chunk capacity
  const int xring = XSTAGED ? 0 : mc;  // activation rows copied per stage
  const int x_slot = xring * kXPitch;

  // layout: codes ring of every warp | x ring of every warp | barriers | tokens
  //         | pre-staged activations | their group sums
  Ring R;
  R.S = S;
  R.x_slot = x_slot;
  constexpr int kSlot = PT ? G::kCodeSlot : G::kSlot;  // PT: the stage boxes carry codes only
  R.codes0 = smem_u32(base) + (uint32_t)(warp * S * kSlot);
  R.xs0 = smem_u32(base) + (uint32_t)(kW * S * kSlot + warp * S * x_slot);
  const uint32_t bar_off = (uint32_t)(kW * ring_bytes<NSUB>(S, xring, PT));
  R.bars0 = smem_u32(base) + bar_off + (uint32_t)(warp * S * 8);
  int* s_tok = reinterpret_cast<int*>(base + bar_off + kW * S * 8);
  const uint32_t xst = smem_u32(base) + bar_off + (uint32_t)(kW * S * 8 + kStreamMisc);  // 16-byte aligned
  const uint32_t sxs = xst + (uint32_t)(mc * p.xpitch);
  int* s_tab = reinterpret_cast<int*>(base + (xst - smem_u32(base)));  // routed mode: chunk table
  R.issued = R.consumed = 0;
  R.pol_stream = policy_evict_first();
  R.pol_keep = policy_evict_last();
  if (p.wait_limit) R.limit = p.wait_limit;
  // G128 / PT: a unit's scales and biases (its rows over the whole K) arrive
  // with its first stage, into one of S slots per warp (a unit has at least
  // one stage, so at most S units are in flight).  G128: K / 64 bytes a row.
  // PT (K % 512 != 0, no tensor map takes rows K / 32 bytes apart): K / 32
  // bytes a row, each table at the same offset modulo 16 as in memory, with
  // room for the 16-byte reads of the last stage that run past the last row
  // (up to 14 + 31 K/32 + 16 ceil(K / 512) < 32 K/32 + 30 bytes).
  const uint32_t prb = (uint32_t)(G128 ? p.K / 64 : p.K / 32);
  const uint32_t phalf = G128 ? kRows * prb : (kRows * prb + 45) & ~15u;
  const uint32_t pslot = 2u * phalf;
  const uint32_t par0 = smem_u32(base) + (uint32_t)p.par_off + (uint32_t)(warp * S) * pslot;
  const uint32_t plow = prb & (0u - prb);       // largest power of two dividing the PT row pitch
  const uint32_t pal = plow < 8u ? plow : 8u;  // the alignment of every PT parameter read
  const int gv_last = p.K / kGroup - 8 * (p.nst - 1);                 // groups inside K in the last stage

  if (lane == 0)
    for (int i = 0; i < S; ++i) mbar_init(R.bars0 + 8 * i, 1);
  if (!ROUTED && threadIdx.x < mc) s_tok[threadIdx.x] = p.row0 + threadIdx.x;
  const uint32_t xbar = smem_u32(s_tok + kMaxChunk + 8 * 8);  // the pre-staged activations' copy
  if (XSTAGED && threadIdx.x == 0) mbar_init(xbar, 1);
  unsigned long long* s_best =  // [warp][8]; the offset is a multiple of 8
      reinterpret_cast<unsigned long long*>(base + (xst - smem_u32(base)) +
                                            (XSTAGED ? xstage_bytes(mc, p.nst * kStageK) : 0));
  unsigned long long* s_cta_best = s_best + 8 * 8;
  if (ARGMAX && threadIdx.x < 8 * 8 + 8) s_best[threadIdx.x] = 0ull;
  int* s_grab = s_tok + kMaxChunk + 8 * 8 + 2;  // the CTA's own unit counter (no workspace)
  if (threadIdx.x == 0) *s_grab = 0;
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();

  // warp-major numbering: the first pass over the units spreads them evenly over CTAs
  const int gw = warp * gridDim.x + blockIdx.x;
  const int TW = gridDim.x * kW;
  // dealing inside the CTA (no workspace): its range, first unit and stride
  const bool own = !ROUTED && local;
  const int cta_lo = own ? (int)((int64_t)blockIdx.x * p.units / gridDim.x) : 0;
  const int cta_hi = own ? (int)((int64_t)(blockIdx.x + 1) * p.units / gridDim.x) : p.units;
  const int first_u = own ? cta_lo + warp : gw;

  // Work units of this warp.  The first is static (unit gw), so its weights
  // can be requested before the wait for earlier kernels.  With DYN every
  // later one is grabbed from a counter in the workspace (unit TW + count)
  // when at most `lead` stages of the previous one are left to request, so warps
  // that run faster take more units and no warp commits to a unit long
  // before it can start it; otherwise the warp takes units gw + TW, ...
  // Lane 0 streams the units in order; dealt ones it records in s_units (a
  // ring of 8 per warp, ahead of the computing lanes by at most S stages;
  // -1 marks the end).
  //
  // Every warp with a first unit grabs until one grab fails, so a launch
  // makes exactly max(0, units - TW) + min(TW, units) grabs; the one that
  // draws the last count resets the counter for the next launch.  A grab's
  // count is only looked at when its unit begins, a stage or two later, so
  // the atomic's round trip does not stall the warp.  Dealt inside the CTA
  // the same happens with the CTA's range and a shared-memory counter,
  // which needs no reset.
  int* s_units = s_tok + kMaxChunk + 8 * warp;
  int units = p.units;             // routed mode: set from the chunk table
  int iu = -1, ist = 0, iend = 0;  // lane 0: unit being issued, its stage cursor
  const int* itok = s_tok;         // lane 0: activation rows of unit iu
  int imc = xring;                 // and their count
  int nxt = -1;                    // lane 0: count of the grab for the unit after iu (unit TW + nxt), -1 before it
  int irow = 0;                    // lane 0: first weight row of unit iu
  int irows = 0;                   // lane 0: and its rows inside the matrix
  int ifirst = 0;                  // lane 0: first stage of unit iu
  uint32_t iseq = 0, ipar = 0;     // lane 0: units dealt / begun
  const int last_grab = max(0, p.units - TW) + min(TW, p.units) - 1;
  // Stages of the current unit still to request when the next is grabbed:
  // one, or two for units of three stages or fewer (LM head 262144x1536:
  // 41.8 -> 41.5 us; one is best from five stages on: 262144x2560, 16384^2).
  const int lead = p.sl <= 3 ? 2 : 1;
  auto grab = [&]() { return own ? atomicAdd(s_grab, 1) : atomicAdd(p.sched, 1); };
  auto resolve = [&](int c) {  // the unit of grab count c, -1 past the end
    if (own) {
      const int v = cta_lo + kW + c;
      return v < cta_hi ? v : -1;
    }
    if (c == last_grab) *p.sched = 0;
    const int v = TW + c;
    return v < p.units ? v : -1;
  };
  auto begin_unit = [&](int u) {
    iu = u;
    if (DYN) s_units[iseq++ & 7u] = u;
    if (UBLK && u >= 0) ++ipar;
    if (u >= 0) {
      if (ROUTED) {
        const int c = u / p.tiles;
        const int* ch = s_tab + 2 + c * (2 + kMaxChunk);
        irow = ch[0] * p.N + (u - c * p.tiles) * kRows;  // row of the stacked [E][N] weights
        irows = min(kRows, p.N - (u - c * p.tiles) * kRows);
        imc = ch[1];
        itok = ch + 2;
        ist = 0;
        iend = p.nst;
      } else if (WHOLEK || G128 || (PT && !SPLIT)) {
        irow = u * kRows;
        irows = min(kRows, p.N - irow);
        ist = 0;
        iend = p.nst;
      } else {
        int slice;
        irow = unit_tile<SPLIT>(p, u, slice) * kRows;
        irows = min(kRows, p.N - irow);  // PT: a split unit brings its rows over the whole K
        ist = slice * p.sl;
        iend = min(ist + p.sl, p.nst);
      }
      ifirst = ist;
    }
  };
  auto issue_stage = [&](bool with_x) {
    uint32_t slot;
    if (UBLK) {
      slot = R.issued % (uint32_t)R.S;
      const uint32_t dst = R.codes0 + slot * kSlot, bar = R.bars0 + 8 * slot;
      if (PT && ist == ifirst) {
        // The unit's rows are bytes [b0, b1) of the scales and of the biases.
        // The 16-byte-aligned window around them comes by one bulk copy per
        // table (byte b to ps + b - lo), clipped at the arrays' last whole 16
        // bytes; bytes past that by plain loads, stored before the barrier is
        // armed (its arrival releases them to the computing lanes).
        const char* gs = reinterpret_cast<const char*>(p.S);
        const char* gb = reinterpret_cast<const char*>(p.B);
        const int64_t tot = (int64_t)(ROUTED ? p.E : 1) * p.N * prb;
        const int64_t b0 = (int64_t)irow * prb, b1 = b0 + (int64_t)irows * prb;
        const int64_t lo = b0 & ~(int64_t)15;
        const int64_t hi = min((b1 + 15) & ~(int64_t)15, tot & ~(int64_t)15);
        const uint32_t nb = hi > lo ? (uint32_t)(hi - lo) : 0u;
        const uint32_t ps = par0 + ((ipar - 1) % (uint32_t)S) * pslot;
        for (int64_t o = max(hi, b0); o < b1; o += 2) {
          const uint16_t vs = ld_nc_u16(reinterpret_cast<const uint16_t*>(gs + o));
          const uint16_t vb = ld_nc_u16(reinterpret_cast<const uint16_t*>(gb + o));
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(ps + (uint32_t)(o - lo)), "h"(vs) : "memory");
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(ps + phalf + (uint32_t)(o - lo)), "h"(vb) : "memory");
        }
        issue_weights<NSUB, false>(dst, 0, bar, &maps, ist, irow, imc, R.pol_stream, R.pol_keep, 2 * nb,
                                   ist * kStageWords + kBoxWords < p.K / 8);
        if (nb) {
          bulk_load(ps, gs + lo, nb, bar, R.pol_keep);
          bulk_load(ps + phalf, gb + lo, nb, bar, R.pol_keep);
        }
      } else if (ist == ifirst) {
        // the unit's rows of the group-128 scales and biases: one bulk copy
        // each of the 16-byte multiple, plain loads for the few bytes past it
        const int rows = min(kRows, p.N - irow);
        const uint32_t nbytes = (uint32_t)rows * prb, bulk = nbytes & ~15u;
        const uint32_t ps = par0 + ((ipar - 1) % (uint32_t)S) * pslot;
        issue_weights<NSUB, false>(dst, 0, bar, &maps, ist, irow, imc, R.pol_stream, R.pol_keep, 2 * bulk);
        const char* gs = reinterpret_cast<const char*>(p.S) + (int64_t)irow * prb;
        const char* gb = reinterpret_cast<const char*>(p.B) + (int64_t)irow * prb;
        if (bulk) {
          bulk_load(ps, gs, bulk, bar, R.pol_keep);
          bulk_load(ps + kRows * prb, gb, bulk, bar, R.pol_keep);
        }
        for (uint32_t o = bulk; o < nbytes; o += 2) {
          const uint16_t vs = ld_nc_u16(reinterpret_cast<const uint16_t*>(gs + o));
          const uint16_t vb = ld_nc_u16(reinterpret_cast<const uint16_t*>(gb + o));
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(ps + o), "h"(vs) : "memory");
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(ps + kRows * prb + o), "h"(vb) : "memory");
        }
      } else {
        issue_weights<NSUB, false>(dst, 0, bar, &maps, ist, irow, imc, R.pol_stream, R.pol_keep, 0,
                                   !PT || ist * kStageWords + kBoxWords < p.K / 8);
      }
      ++R.issued;
    } else {
      const bool fault = p.fault_tx && blockIdx.x == 0 && warp == 0 && R.issued == 0;
      slot = ring_issue_w<NSUB>(R, &maps, ist, irow, imc, fault ? (uint32_t)p.fault_tx : 0u);
    }
    if (with_x) ring_issue_x(R, slot, ist, p.x, itok, imc, p.K);
    ++ist;
  };
  auto issue_next = [&](bool with_x) {  // after the wait only (grabs touch the workspace)
    if (iu < 0) return;
    if (ist == iend) {
      if (DYN) {
        begin_unit(resolve(nxt));
        nxt = -1;
      } else if (own) {
        begin_unit(iu + kW < cta_hi ? iu + kW : -1);
      } else {
        begin_unit(iu + TW < units ? iu + TW : -1);
      }
      if (iu < 0) return;
    }
    issue_stage(with_x);
    if (DYN && nxt < 0 && iend - ist <= lead) nxt = grab();
  };
  // The weights never depend on earlier kernels: with p.prefetch the first
  // unit's first stages are requested before the wait for those kernels and
  // their activation chunks after it.  Activations, outputs and the
  // workspace are only touched after the wait.  The first stages stay in
  // flight while the activations are staged.
  if (lane == 0) {
    fence_proxy_async();
    if (!ROUTED) {
      begin_unit(first_u < cta_hi ? first_u : -1);
      if (p.prefetch)
        for (int i = 0; i < S && iu >= 0 && ist < iend; ++i) issue_stage(false);
    } else if (p.l2_stages > 0) {
      // Routed: which experts are read is known only after the wait for the
      // kernel that wrote the ids.  Until then the grid pulls the first
      // l2_stages stages of every expert's tiles into L2 (a bounded budget;
      // the bytes of experts no token selects are read for nothing).
      const int per_e = p.tiles * p.l2_stages, total = p.E * per_e;
      for (int k = gw; k < total; k += TW) {
        const int e = k / per_e, r = k - e * per_e, tile = r / p.l2_stages, st = r - tile * p.l2_stages;
        const int row = e * p.N + tile * kRows;
        tma_prefetch_l2(&maps.codes, st * kStageWords, row);
        tma_prefetch_l2(&maps.codes, st * kStageWords + kBoxWords, row);
        tma_prefetch_l2(&maps.scales, st * 8, row);
        tma_prefetch_l2(&maps.biases, st * 8, row);
      }
    }
  }
  pdl_wait();
  if (ROUTED) {
    // the chunks the ids select (the same table in every CTA); the first
    // CTA also writes zero rows for tokens whose id is out of range
    if (warp == 0) build_chunks(p.ids, p.T, p.E, mc, s_tab);
    __syncthreads();
    units = s_tab[0] * p.tiles;
    if (blockIdx.x == 0 && s_tab[1] > 0) {
      const int* bad = s_tab + 2 + p.T * (2 + kMaxChunk);
      if (threadIdx.x == 0) atomicOr(p.flags, W4A16_DEVICE_BAD_ID);
      for (int64_t i = threadIdx.x; i < (int64_t)s_tab[1] * p.N; i += blockDim.x)
        p.y[(int64_t)bad[i / p.N] * p.N + i % p.N] = 0;
    }
    if (lane == 0) begin_unit(gw < units ? gw : -1);
  }
  if (XSTAGED && threadIdx.x == 0) {  // each activation row in one bulk copy (16-byte aligned: K % 64 == 0)
    const int kp = p.nst * kStageK;  // then zeros up to the padded K
    mbar_expect_tx(xbar, (uint32_t)(mc * 2 * kp));
    for (int n = 0; n < mc; ++n) {
      bulk_load(xst + n * p.xpitch, p.x + (int64_t)(p.row0 + n) * p.K, 2 * p.K, xbar, R.pol_keep);
      if (kp > p.K) bulk_load(xst + n * p.xpitch + 2 * p.K, g_xzero, 2 * (kp - p.K), xbar, R.pol_keep);
    }
  }
  if (lane == 0) {
    if (iu >= 0) {
      if (DYN && iend - ist <= lead) nxt = grab();
      const int first = ist - (int)R.issued;  // the unit's first stage
      for (uint32_t i = 0; i < R.issued; ++i) ring_issue_x(R, i, first + (int)i, p.x, s_tok, xring, p.K);
    }
    for (int i = (int)R.issued; i < S; ++i) issue_next(true);
  }
  __syncwarp();

  bool timed_out = false;
  if (XSTAGED) {
    // Activation rows in B-fragment order and the sum of every 64-group of
    // every row, from one bulk copy per row.  The copy goes out through the
    // tensor-memory-access path, which returns it well ahead of per-thread
    // loads while the first weight stages are in flight.
    timed_out = __syncthreads_or(!mbar_wait(xbar, 0)) != 0;
    // One pass over the staged rows: every 16-byte chunk is read, put in
    // B-fragment order in registers and written back in place, and the same
    // registers feed the group sums.  One MMA chain yields eight groups of
    // one activation row, the group in the MMA column (lane (g, t) holds
    // chunks t and 4 + t of group g, which together cover every chunk once).
    // An output column depends only on its own B column, so every sum has
    // the bits of the per-stage chain (activation row in the column).  Four
    // chains per warp at a time, interleaved.
    const int nblk = p.nst, tasks = timed_out ? 0 : mc * nblk;
    for (int k0 = warp; k0 < tasks; k0 += 4 * kW) {
      uint32_t b[4][2][2][2];
      float v[4][4];
      uint4 raw[4][2];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int k = k0 + j * kW;
        const int n = k / nblk, blk = k - n * nblk;
#pragma unroll
        for (int cb = 0; cb < 2; ++cb)
          raw[j][cb] = k < tasks ? lds128(xst + n * p.xpitch + 128 * (8 * blk + g) + 64 * cb + 16 * t)
                                 : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int k = k0 + j * kW;
        const int n = k / nblk, blk = k - n * nblk;
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
          frag_from_chunk(raw[j][cb], b[j][cb]);
          if (k < tasks)
            sts128(xst + n * p.xpitch + 128 * (8 * blk + g) + 64 * cb + 16 * t,
                   make_uint4(b[j][cb][0][0], b[j][cb][0][1], b[j][cb][1][0], b[j][cb][1][1]));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) v[j][i] = 0.f;
      }
#pragma unroll
      for (int step = 0; step < 4; ++step)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          mma_bf16(v[j], kOnes, kOnes, kOnes, kOnes, b[j][step >> 1][step & 1][0], b[j][step >> 1][step & 1][1]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int k = k0 + j * kW;
        const int n = k / nblk, blk = k - n * nblk;
        if (g == 0 && k < tasks) {  // row 0 of D: columns 2t, 2t+1 are groups 8 blk + 2t, + 1
          const int gi = 8 * blk + 2 * t;
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(sxs + (gi * sx_cols(mc) + n) * 4), "f"(v[j][0]) : "memory");
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(sxs + ((gi + 1) * sx_cols(mc) + n) * 4), "f"(v[j][1])
                       : "memory");
        }
      }
    }
    __syncthreads();
  }
  uint32_t loff2[2][4];
  ldsm_offsets(lane, loff2);
  uint32_t loff[NSUB][4];
#pragma unroll
  for (int s = 0; s < NSUB; ++s)
#pragma unroll
    for (int i = 0; i < 4; ++i) loff[s][i] = loff2[s][i];

  int pend_tile = -1;               // partials stored, arrival not yet counted
  int cnt_tile = -1, cnt_old = 0;   // arrival counted (lane 0 holds the old count)

  auto reduce_tiles = [&](int ta, int tb) {
    // Sum the ksplit partials of finished tiles ta and tb (-1: none) in
    // slice order.  Lane 0's fence (after it saw the last arrivals) and the
    // warp barrier order every lane's loads after the other units' partial
    // stores.  Loads are issued eight slices of both tiles at a time; the
    // additions stay in slice order.
    if (lane == 0) fence_acq_rel_gpu();
    __syncwarp();
    // lane = (column n0, row r): with 16 rows two columns at a time
    const int r = lane % kRows, n0 = lane / kRows;
    const int tt[2] = {ta, tb};
    for (int n = n0; n < mc; n += 32 / kRows) {
      float sum[2] = {0.0f, 0.0f};
      for (int s0 = 0; s0 < p.ks; s0 += 8) {
        float v[2][8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float* q = p.part + ((int64_t)max(tt[h], 0) * p.ks * 8 + n) * kRows + r;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            v[h][j] = (tt[h] >= 0 && s0 + j < p.ks) ? __ldcg(q + (int64_t)(s0 + j) * 8 * kRows) : 0.0f;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (s0 + j < p.ks) sum[h] = (s0 + j == 0) ? v[h][0] : __fadd_rn(sum[h], v[h][j]);
      }
      if (ARGMAX) {
        unsigned long long k = 0ull;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = tt[h] * kRows + r;
          if (tt[h] >= 0 && row < p.N) k = max_u64(k, argmax_key(f32_to_bf16_bits(sum[h]), row));
        }
        k = warp_max_u64(k, 16, 1);  // the 32 rows of the tile
        if (lane == 0) s_best[warp * 8 + n] = max_u64(s_best[warp * 8 + n], k);
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = tt[h] * kRows + r;
          if (tt[h] >= 0 && row < p.N) p.y[(int64_t)s_tok[n] * p.N + row] = f32_to_bf16_bits(sum[h]);
        }
      }
    }
    if (lane == 0) {
      if (ta >= 0) p.cnt[ta] = 0;
      if (tb >= 0) p.cnt[tb] = 0;
    }
  };
  auto reduce_tile = [&](int tile) { reduce_tiles(tile, -1); };

  // Count the arrival of this warp's stored partials of `tile`: a warp
  // barrier, then one release fence by lane 0 before its atomic.
  auto count_arrival = [&](int tile) {
    __syncwarp();
    if (lane == 0) {
      fence_acq_rel_gpu();
      cnt_old = atomicAdd(p.cnt + tile, 1);
    }
    cnt_tile = tile;
  };

  auto rows_of = [&](int tile, int (&pr)[2 * NSUB]) {
#pragma unroll
    for (int i = 0; i < 2 * NSUB; ++i) pr[i] = tile * kRows + 16 * (i >> 1) + g + 8 * (i & 1);
  };

  // consume cursor: round-robin units follow from gw; dealt ones are read
  // in the order lane 0 recorded them
  int u = first_u;
  for (uint32_t cseq = 0; !timed_out; ++cseq) {
    if (DYN) {
      __syncwarp();
      u = s_units[cseq & 7u];
    } else if (cseq > 0) {
      u += own ? kW : TW;
    }
    if (u < 0 || u >= (own ? cta_hi : units)) break;
    int slice = 0, tile, umc = mc;
    const int* utok = s_tok;
    int64_t crow;  // the unit's first row in the (stacked) weights
    if (ROUTED) {
      const int c = u / p.tiles;
      const int* ch = s_tab + 2 + c * (2 + kMaxChunk);
      tile = u - c * p.tiles;
      umc = ch[1];
      utok = ch + 2;
      crow = (int64_t)ch[0] * p.N + tile * kRows;
    } else {
      tile = unit_tile<SPLIT>(p, u, slice);
      crow = (int64_t)tile * kRows;
    }
    // PT: the unit's parameter rows in its slot, at their offset modulo 16
    const uint32_t ppar = par0 + (cseq % (uint32_t)S) * pslot + (uint32_t)((crow * prb) & 15);
    const int s0 = FOLD ? 0 : slice * p.sl, s1 = FOLD ? p.nst : min(s0 + p.sl, p.nst);
    // The last slice of a tile reads the tile's arrival count before its
    // stages (the value is used after them, so the load never stalls).
    const bool last_slice = SPLIT && slice == p.ks - 1;
    int seen = 0;
    if (last_slice && lane == 0) seen = ld_relaxed_gpu(p.cnt + tile);
    int prow[2 * NSUB];
    rows_of(tile, prow);

    float acc[NSUB][4];
#pragma unroll
    for (int s = 0; s < NSUB; ++s)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[s][i] = 0.0f;
    float sum[NSUB][4];       // whole-K units: the slice sums folded so far, in slice order
    int fold_at = s0 + p.sl;  // and the stage that ends the current slice

    for (int st = s0; st < s1; ++st) {
      uint32_t slot;
      if (!ring_wait(R, slot)) {
        timed_out = true;
        break;
      }
      const uint32_t cbase = ordered(R.codes0 + slot * kSlot);
      uint32_t xbase, sxbase = 0;
      if (XSTAGED) {
        xbase = xst + g * p.xpitch + 16 * t + st * (kStageK * 2);
        sxbase = sxs + (st * (kStageK / kGroup) * sx_cols(mc) + 2 * t) * 4;
      } else {
        xbase = ordered(R.xs0 + slot * x_slot + g * kXPitch + 16 * t);
      }
      if (G128)
        compute_stage_sel<NSUB, ALLCOLS, XSTAGED, 16 * NSUB, 1>(
            cbase, par0 + (cseq % (uint32_t)S) * pslot + (uint32_t)st * 8u, xbase, g < umc, sxbase, sx_cols(mc) * 4,
            2 * t < umc, acc, loff, g, prb, kRows * prb);
      else if (PT)
        compute_stage_sel<NSUB, ALLCOLS, XSTAGED, 16 * NSUB, 2>(
            cbase, ppar + (uint32_t)st * 16u, xbase, g < umc, sxbase, sx_cols(mc) * 4, 2 * t < umc, acc, loff, g,
            prb, phalf, pal, st == p.nst - 1 ? gv_last : 8);
      else
        compute_stage_sel<NSUB, ALLCOLS, XSTAGED>(cbase, cbase + 2 * G::kBox, xbase, g < umc, sxbase,
                                                  sx_cols(mc) * 4, 2 * t < umc, acc, loff, g);
      if (FOLD && (st + 1 == fold_at || st + 1 == s1)) {
        const bool first = fold_at == s0 + p.sl;
#pragma unroll
        for (int s = 0; s < NSUB; ++s)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            sum[s][i] = first ? acc[s][i] : __fadd_rn(sum[s][i], acc[s][i]);
            acc[s][i] = 0.0f;
          }
        fold_at += p.sl;
      }
      ++R.consumed;
      __syncwarp();
      if (lane == 0) {
        fence_proxy_async();
        issue_next(true);
      }
    }
    if (timed_out) break;

    // Split-K arrivals run two units behind the stores: the arrival counted
    // one unit ago has had a whole unit to come back, and the partials
    // stored one unit ago have had a whole unit to land, so neither the
    // fence nor the atomic stalls the warp.
    if (cnt_tile >= 0) {
      const int old = __shfl_sync(0xffffffffu, cnt_old, 0);
      if (old == p.ks - 1) reduce_tile(cnt_tile);
      cnt_tile = -1;
    }
    if (pend_tile >= 0) {
      count_arrival(pend_tile);
      pend_tile = -1;
    }
    if (FOLD) {  // routed rows go to their tokens; plain rows to row0 + n
#pragma unroll
      for (int s = 0; s < NSUB; ++s)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = prow[2 * s + (i >> 1)];
          const int n = 2 * t + (i & 1);
          if (n < umc && row < p.N) p.y[(int64_t)utok[n] * p.N + row] = f32_to_bf16_bits(sum[s][i]);
        }
    } else if (!SPLIT && ARGMAX) {
      // columns 2t and 2t + 1: the lane's rows, then the eight lanes of t
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int n = 2 * t + c;
        unsigned long long k = 0ull;
#pragma unroll
        for (int s = 0; s < NSUB; ++s)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int row = prow[2 * s + rr];
            if (row < p.N) k = max_u64(k, argmax_key(f32_to_bf16_bits(acc[s][2 * rr + c]), row));
          }
        k = warp_max_u64(k, 16, 4);
        if (g == 0 && n < mc) s_best[warp * 8 + n] = max_u64(s_best[warp * 8 + n], k);
      }
    } else if (!SPLIT) {
#pragma unroll
      for (int s = 0; s < NSUB; ++s)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = prow[2 * s + (i >> 1)];
          const int n = 2 * t + (i & 1);
          if (n < mc && row < p.N) p.y[(int64_t)s_tok[n] * p.N + row] = f32_to_bf16_bits(acc[s][i]);
        }
    } else {
      float* q = p.part + ((int64_t)tile * p.ks + slice) * 8 * kRows;
#pragma unroll
      for (int s = 0; s < NSUB; ++s)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 16 * s + g + 8 * (i >> 1);
          const int n = 2 * t + (i & 1);
          if (n < mc) __stcg(q + n * kRows + r, acc[s][i]);
        }
      // A last slice that found every other slice arrived adds the tile up at
      // once: reduce_tile's fence by lane 0 (after it read the count) and warp
      // barrier order the loads after the others' partial stores and this
      // warp's own.  Nobody else touches the count in this launch.
      if (last_slice && __shfl_sync(0xffffffffu, seen, 0) == p.ks - 1)
        reduce_tile(tile);
      else
        pend_tile = tile;
    }
  }
  if (!timed_out) {
    // The tile counted one unit ago and this warp's last one: both arrivals
    // are known before either sum, so their loads go out together.
    int prev = -1, last = -1;
    if (cnt_tile >= 0 && __shfl_sync(0xffffffffu, cnt_old, 0) == p.ks - 1) prev = cnt_tile;
    if (pend_tile >= 0) {
      count_arrival(pend_tile);
      if (__shfl_sync(0xffffffffu, cnt_old, 0) == p.ks - 1) last = pend_tile;
    }
    if (prev >= 0 || last >= 0) reduce_tiles(prev, last);
  }
  if (timed_out) {
    if (lane == 0) atomicOr(p.flags, W4A16_DEVICE_TIMEOUT);
    // finish this warp's grabs (up to the one that fails), so the count of
    // grabs stays exact and the counter is reset
    if (DYN && !own && lane == 0 && iu >= 0)
      for (int v = nxt >= 0 ? resolve(nxt) : 0; v >= 0; v = resolve(grab())) {
      }
    // let copies already in flight land before shared memory is released
    if (XSTAGED) mbar_wait(xbar, 0);
    const uint32_t issued = __shfl_sync(0xffffffffu, R.issued, 0);
    while (R.consumed < issued) {
      mbar_wait(R.bars0 + 8 * (R.consumed % (uint32_t)S), (R.consumed / (uint32_t)S) & 1u);
      ++R.consumed;
    }
  }
  if (ARGMAX) {
    // this warp's keys into the CTA's, the CTA's into the launch's; the last
    // CTA out (every CTA fences its atomics before counting itself) turns
    // the keys into indices and values and leaves both counters at zero
    __syncwarp();
    if (lane < mc) atomicMax(s_cta_best + lane, s_best[warp * 8 + lane]);
    __syncthreads();
    if (threadIdx.x < mc) {
      atomicMax(p.best + threadIdx.x, s_cta_best[threadIdx.x]);
      __threadfence();
    }
    __syncthreads();
    int* s_last = reinterpret_cast<int*>(s_cta_best);  // the CTA's keys are merged by now
    if (threadIdx.x == 0) {
      __threadfence();
      *s_last = atomicAdd(p.done, 1) == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (*s_last && threadIdx.x < mc) {  // one thread per activation row
      __threadfence();
      const int n = threadIdx.x;
      const unsigned long long k = atomicExch(p.best + n, 0ull);
      const uint32_t ord = (uint32_t)(k >> 32);
      p.idx[p.row0 + n] = (int32_t)(0xFFFFFFFFu - (uint32_t)k);
      if (p.val) p.val[p.row0 + n] = (uint16_t)((ord & 0x8000u) ? (ord & 0x7FFFu) : (~ord & 0xFFFFu));
      if (n == 0) *p.done = 0;
    }
  }
}

// ---- tile kernel (w4a16_mm when every warp would get about one unit) ---------------------
//
// A 16-row tile's K range is split over a cluster of kc CTAs (kc = 1: one
// CTA); each CTA holds its share in shared memory at once, one slot per
// 512-code stage, all requested up front.  Warp w of a CTA computes its
// slices w, w + W, ... (one m16 subtile), so a warp's serial work is a single
// 16-row slice.  Every slice sum goes to the shared memory of the cluster's
// first CTA (distributed shared memory), which adds them in slice order --
// the same canonical arithmetic as the persistent kernel, with no workspace,
// atomics or global fences.

constexpr int kTile16 = Geo<1>::kRows;
constexpr int kTileMaxWarps = 16;
constexpr int kMaxCluster = 8;

// Operands of the tile kernel per item: one item for w4a16_mm and
// w4a16_mm_id, up to kMaxGroup for w4a16_mm_group (items share K, M and
// hence the slicing).
constexpr int kMaxGroup = W4A16_MAX_GROUP;
template <int G>
struct TileArgs {
  Maps maps[G];
  const uint16_t* S[G];  // the parameter tables (read by bulk copy with K % 512 != 0)
  const uint16_t* B[G];
  const uint16_t* x[G];
  uint16_t* y[G];
  int N[G];
  int tile0[G + 1];  // first 16-row tile of item i in the grid; tile0[items] = all tiles
};

struct TileParams {
  int* flags;
  const int32_t* ids;  // routed mode: expert id per token
  int items;           // items in TileArgs
  int K, M, row0;      // plain mode: rows row0 .. row0 + M of x, xcap at a time
  int T, E;            // routed mode: tokens, experts
  int nst, sl, ks;
  int kc;        // CTAs (one cluster) per 16-row tile
  int nloc;      // stage slots per CTA: ceil(ks / kc) * sl
  int xcap;      // activation rows per x slot (plain: M; routed: tokens per chunk)
  int prefetch;  // request the weights before waiting for earlier kernels
};

// Shared memory (the same layout in every CTA of a cluster): codes
// [nloc][4096 R] | scales and biases [nloc][512 R] | activation chunks
// [nloc][xcap][kXPitch] | barriers [nloc] | slice sums [ks][16 R][xcap] fp32
// (used in the first CTA) | tokens [8], abort flag, token-scan state [2].
// R = 1 or 2 m16 row subtiles per CTA (16 or 32 rows): with R = 2 two warps,
// one per subtile, share every stage's activation chunk.
// ptK (K % 512 != 0, else 0): the stages carry codes only, and the CTA's
// parameter rows (16 R rows over the whole K, scales then biases, each in
// tile_pt_half bytes) follow the rest at the next 16-byte boundary.
__host__ __device__ inline int tile_pt_half(int K, int R) { return (16 * R * (K / 32) + 45) & ~15; }
__host__ __device__ inline int tile_smem_body(int nloc, int xcap, int ks, int R, bool pt) {
  return nloc * (R * (2 * Geo<1>::kBox + (pt ? 0 : 2 * Geo<1>::kParam)) + xcap * kXPitch) + nloc * 8 +
         ks * kTile16 * R * xcap * 4 + 64;
}
__host__ __device__ inline int tile_smem(int nloc, int xcap, int ks, int R = 1, int ptK = 0) {
  const int body = tile_smem_body(nloc, xcap, ks, R, ptK != 0);
  return (ptK ? ((body + 15) & ~15) + 2 * tile_pt_half(ptK, R) : body) + 1024;
}

__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Plain mode (w4a16_mm): blockIdx.x = tile * kc + rank; the M rows go through
// in chunks of xcap (at most eight) while the weights stay in shared memory,
// so a launch reads them once for any M.
// Routed mode (w4a16_mm_id): blockIdx.y = expert e.  After the wait for
// earlier kernels every CTA collects, in token order, the tokens routed to e
// (at most xcap at a time) and exits when there are none, so an untouched
// expert's weights are never read.  Its weights are requested once and stay
// in shared memory while the token chunks stream through; the CTAs of e = 0
// also write zero rows for tokens whose id is out of range and raise the
// flag.  Every row's arithmetic is the canonical one, so routed rows equal
// w4a16_mm on the selected expert bit for bit.
//
// The bound of 768 threads caps registers at 80, so that five CTAs of five
// warps fit on an SM (by registers).
// MULTI: more activation rows than one chunk (M > xcap); a separate instance,
// so that one-chunk launches carry none of the loop's code.
// PT: K % 512 != 0 (K padded to whole stages): the stages carry codes only
// and the CTA's parameter rows come by bulk copy with its first stage, as in
// the persistent kernel's PT mode.
template <bool ALLCOLS, bool ROUTED, int G, int R, bool MULTI = false, bool PT = false>
__global__ void __launch_bounds__(768) tc_tile_kernel(const __grid_constant__ TileArgs<G> ta, TileParams p) {
  static_assert(!PT || G == 1, "K % 512 != 0: single matrices");
  constexpr int kRowsR = 16 * R, kCodesR = 2 * R * Geo<1>::kBox, kParamsR = PT ? 0 : 2 * R * Geo<1>::kParam;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, W = blockDim.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int kc = p.kc;
  // with cluster dimensions (kc, 1, 1) the rank in the cluster is blockIdx.x % kc
  const int tile_g = blockIdx.x / kc, crank = blockIdx.x - tile_g * kc;
  int item = 0;
  if (G > 1)
    while (item + 1 < p.items && tile_g >= ta.tile0[item + 1]) ++item;
  const int tile = tile_g - ta.tile0[item];
  const Maps& maps = ta.maps[item];
  const uint16_t* __restrict__ xin = ta.x[item];
  uint16_t* __restrict__ yout = ta.y[item];
  const int N = ta.N[item];
  const int j0 = crank * p.ks / kc, j1 = (crank + 1) * p.ks / kc;  // this CTA's slices
  const int st0 = j0 * p.sl, nloc = min(j1 * p.sl, p.nst) - st0;  // and stages
  const int e = ROUTED ? (int)blockIdx.y : 0;
  const int tile_row = tile * kRowsR;
  const int tensor_row = e * N + tile_row;  // row of the stacked [E][N] weights
  const int x_slot = p.xcap * kXPitch, xcap = p.xcap;
  const uint32_t codes0 = smem_u32(base);
  const uint32_t params0 = codes0 + (uint32_t)(p.nloc * kCodesR);
  const uint32_t xs0 = params0 + (uint32_t)(p.nloc * kParamsR);
  const uint32_t bars0 = xs0 + (uint32_t)(p.nloc * x_slot);
  float* red = reinterpret_cast<float*>(base + (bars0 - codes0) + p.nloc * 8);
  int* s_tok = reinterpret_cast<int*>(red + p.ks * kRowsR * xcap);
  int* s_abort = s_tok + kMaxChunk;
  int* s_state = s_abort + 1;  // token scan: [0] position, [1] count
  // PT: the CTA's rows are bytes [pb0, pb0 + prows K/32) of the scales and of
  // the biases, kept at their offset modulo 16 (tile_smem)
  const uint32_t prb = (uint32_t)(p.K / 32);
  const uint32_t phalf = (uint32_t)tile_pt_half(p.K, R);
  const uint32_t pblk = codes0 + (uint32_t)((tile_smem_body(p.nloc, xcap, p.ks, R, true) + 15) & ~15);
  const int64_t pb0 = (int64_t)tensor_row * prb;
  const uint32_t plow = prb & (0u - prb);
  const uint32_t pal = plow < 8u ? plow : 8u;
  const int gv_last = p.K / kGroup - 8 * (p.nst - 1);

  for (int i = threadIdx.x; i < nloc; i += blockDim.x) mbar_init(bars0 + 8 * i, 1);
  if (!ROUTED && threadIdx.x < min(p.M, xcap)) s_tok[threadIdx.x] = p.row0 + threadIdx.x;
  if (threadIdx.x == 0) {
    *s_abort = 0;
    s_state[0] = 0;
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();

  // lane 0 of warp w requests local stages w, w + W, ...
  auto weights = [&](int i, int xrows) {
    if (PT) {
      // With local stage 0: the 16-byte-aligned window around the CTA's
      // parameter rows by one bulk copy per table, clipped at the tables'
      // last whole 16 bytes, and bytes past that by plain loads stored
      // before the stage's barrier is armed.
      uint32_t nb = 0;
      int64_t lo = 0;
      const char* gs = reinterpret_cast<const char*>(ta.S[0]);
      const char* gb = reinterpret_cast<const char*>(ta.B[0]);
      if (i == 0) {
        const int64_t tot = (int64_t)(ROUTED ? p.E : 1) * N * prb;
        const int64_t b1 = pb0 + (int64_t)min(kRowsR, N - tile_row) * prb;
        lo = pb0 & ~(int64_t)15;
        const int64_t hi = min((b1 + 15) & ~(int64_t)15, tot & ~(int64_t)15);
        nb = hi > lo ? (uint32_t)(hi - lo) : 0u;
        for (int64_t o = max(hi, pb0); o < b1; o += 2) {
          const uint16_t vs = ld_nc_u16(reinterpret_cast<const uint16_t*>(gs + o));
          const uint16_t vb = ld_nc_u16(reinterpret_cast<const uint16_t*>(gb + o));
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(pblk + (uint32_t)(o - lo)), "h"(vs) : "memory");
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(pblk + phalf + (uint32_t)(o - lo)), "h"(vb) : "memory");
        }
      }
      issue_weights<R, false>(codes0 + i * kCodesR, 0, bars0 + 8 * i, &maps, st0 + i, tensor_row, xrows,
                              policy_evict_first(), policy_evict_last(), 2 * nb,
                              (st0 + i) * kStageWords + kBoxWords < p.K / 8);
      if (nb) {
        bulk_load(pblk, gs + lo, nb, bars0, policy_evict_last());
        bulk_load(pblk + phalf, gb + lo, nb, bars0, policy_evict_last());
      }
    } else {
      issue_weights<R>(codes0 + i * kCodesR, params0 + i * kParamsR, bars0 + 8 * i, &maps, st0 + i, tensor_row,
                       xrows, policy_evict_first(), policy_evict_last());
    }
  };
  if (!ROUTED && lane == 0 && p.prefetch)
    for (int i = warp; i < nloc; i += W) weights(i, min(p.M, xcap));
  pdl_wait();
  // Only now let the next kernel launch: its CTAs then fetch their weights
  // while this one computes, and at most one kernel waits ahead (CTAs
  // launched further ahead would only hold SM resources and slow this one).
  pdl_launch_dependents();

  int mc = min(p.M, xcap);  // rows of the current chunk
  if (ROUTED) {
    if (e == 0 && crank == 0) {
      // tokens whose expert id is out of range: zero rows, raise the flag
      for (;;) {
        const int cnt = gather_tokens(p.ids, p.T, p.E, -1, s_tok, s_state);
        if (cnt == 0) break;
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(p.flags, W4A16_DEVICE_BAD_ID);
        for (int i = threadIdx.x; i < cnt * kRowsR; i += blockDim.x) {
          const int row = tile_row + i % kRowsR;
          if (row < N) yout[(int64_t)s_tok[i / kRowsR] * N + row] = 0;
        }
        __syncthreads();
      }
      if (threadIdx.x == 0) s_state[0] = 0;
      __syncthreads();
    }
    mc = gather_tokens(p.ids, p.T, p.E, e, s_tok, s_state, p.xcap);
    if (mc == 0) return;  // the same for every CTA of the cluster: no cluster barrier has run
  }
  // announce that this CTA runs (its shared memory may now be written by the others)
  if (kc > 1) cluster_arrive_relaxed();
  if (lane == 0)
    for (int i = warp; i < nloc; i += W) {
      if (ROUTED || !p.prefetch) weights(i, mc);
      issue_x(xs0 + i * x_slot, bars0 + 8 * i, st0 + i, xin, s_tok, mc, p.K, policy_evict_last());
    }

  // slice sums go to the first CTA of the cluster, once every CTA of it runs
  uint32_t red_dst = smem_u32(red);
  __syncwarp();  // the cluster barrier instructions are .aligned: whole warps only
  if (kc > 1) {
    red_dst = map_to_rank(red_dst, 0);
    cluster_wait();
  }
  // warp w computes subtile w % R (W is a multiple of R) of slices j0 + w / R, + W / R, ...
  const int sub = R == 1 ? 0 : warp % R;
  uint32_t loff2[2][4];
  ldsm_offsets(lane, loff2);
  uint32_t loff[1][4];
#pragma unroll
  for (int q = 0; q < 4; ++q) loff[0][q] = sub ? loff2[1][q] : loff2[0][q];
  auto cta_sync = [&]() {
    __syncwarp();
    if (kc > 1) {
      cluster_arrive();
      cluster_wait();
    } else {
      __syncthreads();
    }
  };

  uint32_t last_issued = 0;  // the chunk whose copies were requested last
  for (uint32_t chunk = 0;; ++chunk) {
    // every stage barrier completes one phase per chunk (weights + x, then x)
    const uint32_t parity = chunk & 1u;
    bool ok = *s_abort == 0;
    // PT: the parameter rows arrive with local stage 0, but the warps compute
    // their stages in parallel: every warp also waits for stage 0's first
    // phase (the copies, and lane 0's plain stores released by its arrival)
    if (PT && chunk == 0 && ok && !__all_sync(0xffffffffu, mbar_wait(bars0, 0))) ok = false;
    for (int j = j0 + warp / R; j < j1 && ok; j += W / R) {
      float acc[1][4] = {{0.f, 0.f, 0.f, 0.f}};
      const int s1 = min((j + 1) * p.sl, p.nst);
      for (int st = j * p.sl; st < s1; ++st) {
        const int i = st - st0;
        if (!__all_sync(0xffffffffu, mbar_wait(bars0 + 8 * i, parity))) {
          ok = false;
          break;
        }
        const uint32_t cbase = ordered(codes0 + i * kCodesR);
        const uint32_t pbase =
            PT ? ordered(pblk + (uint32_t)(pb0 & 15) + (uint32_t)st * 16u + (uint32_t)(sub * kTile16) * prb)
               : ordered(params0 + i * kParamsR + sub * kTile16 * 16);
        const uint32_t xbase = ordered(xs0 + i * x_slot + g * kXPitch + 16 * t);
        compute_stage<1, ALLCOLS, false, kRowsR, PT ? 2 : 0>(cbase, pbase, xbase, g < mc, 0u, 0u, false, acc, loff,
                                                             g, prb, phalf, pal, st == p.nst - 1 ? gv_last : 8);
      }
      if (!ok) break;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int n = 2 * t + (i & 1);
        if (n < xcap)
          st_cluster_f32(red_dst + 4 * ((j * kRowsR + kTile16 * sub + g + 8 * (i >> 1)) * xcap + n), acc[0][i]);
      }
    }
    if (!ok && lane == 0 && *s_abort == 0) {
      atomicOr(p.flags, W4A16_DEVICE_TIMEOUT);
      *s_abort = 1;
    }
    cta_sync();
    const bool aborted = *s_abort != 0;  // sticky: later chunks skip the work but keep the barriers
    if (crank == 0 && !aborted) {
      for (int i = threadIdx.x; i < kRowsR * mc; i += blockDim.x) {
        const int n = i / kRowsR, r = i - n * kRowsR;
        const int row = tile_row + r;
        if (row < N) {
          float sum = red[r * xcap + n];
          for (int j = 1; j < p.ks; ++j) sum = __fadd_rn(sum, red[(j * kRowsR + r) * xcap + n]);
          yout[(int64_t)s_tok[n] * N + row] = f32_to_bf16_bits(sum);
        }
      }
    }
    // the last chunk (uniform in the cluster)
    if (!ROUTED && (!MULTI || (int)(chunk + 1) * xcap >= p.M)) break;
    __syncthreads();  // s_tok is read above and rewritten below
    if (ROUTED) {
      mc = gather_tokens(p.ids, p.T, p.E, e, s_tok, s_state, p.xcap);
    } else {  // the next xcap rows, while the weights stay resident
      const int c0 = (int)(chunk + 1) * xcap;
      mc = c0 < p.M ? min(xcap, p.M - c0) : 0;
      if (threadIdx.x < mc) s_tok[threadIdx.x] = p.row0 + c0 + threadIdx.x;
      __syncthreads();
    }
    if (mc == 0) break;  // the same in every CTA of the cluster
    // the first CTA has summed this chunk and every warp is done with the x slots
    cta_sync();
    if (!aborted) {
      if (lane == 0)
        for (int i = warp; i < nloc; i += W) {
          fence_proxy_async();
          mbar_expect_tx(bars0 + 8 * i, (uint32_t)(mc * kStageK * 2));
          issue_x(xs0 + i * x_slot, bars0 + 8 * i, st0 + i, xin, s_tok, mc, p.K, policy_evict_last());
        }
      last_issued = chunk + 1;
    }
  }
  if (*s_abort && lane == 0) {
    // let every copy this warp requested land before shared memory is released
    for (int i = warp; i < nloc; i += W) mbar_wait(bars0 + 8 * i, last_issued & 1u);
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
  int xcap;  // activation rows per x slot: min(T, 8)
};

__host__ __device__ inline int routed_smem(int warps, int stages, int ks, int xcap) {
  return warps * ring_bytes<2>(stages, xcap) + warps * stages * 8 + ks * kTileRows * 8 * 4 + 16 * 4 + 1024;
}

__global__ void __launch_bounds__(kRoutedWarps * 32) tc_routed_kernel(const __grid_constant__ Maps maps,
                                                                      RoutedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int S = p.stages, W = p.warps;
  const int x_slot = p.xcap * kXPitch;
  const int e = blockIdx.y;
  const int row_base = blockIdx.x * kTileRows;
  const int tensor_row = e * p.N + row_base;

  Ring R;
  R.S = S;
  R.x_slot = x_slot;
  R.codes0 = smem_u32(base) + (uint32_t)(warp * S * kCodeSlotBytes);
  R.xs0 = smem_u32(base) + (uint32_t)(W * S * kCodeSlotBytes + warp * S * x_slot);
  const uint32_t bar_off = (uint32_t)(W * ring_bytes<2>(S, p.xcap));
  R.bars0 = smem_u32(base) + bar_off + (uint32_t)(warp * S * 8);
  float* red = reinterpret_cast<float*>(base + bar_off + W * S * 8);  // [ks][32 rows][8 columns]
  int* s_tok = reinterpret_cast<int*>(red + p.ks * kTileRows * 8);
  int* s_state = s_tok + kMaxChunk;  // [0] scan position, [1] count, [2] abort
  R.issued = R.consumed = 0;
  R.pol_stream = policy_evict_first();
  R.pol_keep = policy_evict_last();

  pdl_launch_dependents();
  if (lane == 0)
    for (int i = 0; i < S; ++i) mbar_init(R.bars0 + 8 * i, 1);
  if (threadIdx.x == 0) {
    s_state[0] = 0;
    s_state[2] = 0;
  }
  pdl_wait();  // ids, activations and outputs belong to earlier kernels
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();

  uint32_t loff[2][4];
  ldsm_offsets(lane, loff);

  // this warp's stages: slices warp, warp + W, ... each [slice*sl, min(nst, ...))
  auto slice_end = [&](int sidx) { return min((sidx + 1) * p.sl, p.nst); };

  for (;;) {
    const int mc = gather_tokens(p.ids, p.T, p.E, e, s_tok, s_state);
    if (mc == 0) break;

    int isl = warp, ist = warp * p.sl;  // issue cursor
    auto issue_next = [&]() {
      if (isl >= p.ks) return;
      ring_issue<2>(R, &maps, ist, tensor_row, p.x, s_tok, mc, p.K);
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
      for (int st = s0; st < s1; ++st) {
        uint32_t slot;
        if (!ring_wait(R, slot)) {
          timed_out = true;
          break;
        }
        const uint32_t cbase = ordered(R.codes0 + slot * kCodeSlotBytes);
        const uint32_t xbase = ordered(R.xs0 + slot * x_slot + g * kXPitch + 16 * t);
        compute_stage<2, true, false>(cbase, cbase + 2 * Geo<2>::kBox, xbase, g < mc, 0u, 0u, false, acc, loff, g);
        ++R.consumed;
        __syncwarp();
        if (lane == 0) {
          fence_proxy_async();
          issue_next();
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
      const uint32_t issued = __shfl_sync(0xffffffffu, R.issued, 0);
      while (R.consumed < issued) {
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

cudaError_t make_param_map(CUtensorMap* map, const uint16_t* P, int64_t rows, int K, int box_rows) {
  if (cudaError_t e = get_encoder()) return e;
  cuuint64_t dims[2] = {(cuuint64_t)(K / kGroup), (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(K / kGroup) * 2};
  cuuint32_t box[2] = {8, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(P), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_code_map(CUtensorMap* map, const uint32_t* Wq, int64_t rows, int K, int box_rows) {
  if (cudaError_t e = get_encoder()) return e;
  cuuint64_t dims[2] = {(cuuint64_t)(K / 8), (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K / 2};
  cuuint32_t box[2] = {(cuuint32_t)kBoxWords, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(Wq), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor maps of one weight set with boxes of box_rows rows (32 for the
// persistent and routed kernels, 16 for the tile kernel).
cudaError_t make_maps(Maps* m, const uint32_t* Wq, const uint16_t* S, const uint16_t* B, int64_t rows, int K,
                      int box_rows = kTileRows) {
  if (cudaError_t e = make_code_map(&m->codes, Wq, rows, K, box_rows)) return e;
  if (cudaError_t e = make_param_map(&m->scales, S, rows, K, box_rows)) return e;
  return make_param_map(&m->biases, B, rows, K, box_rows);
}

template <int NSUB>
int stream_smem(int stages, int mc, bool codes_only = false) {
  using G = Geo<NSUB>;
  return G::kWarps * ring_bytes<NSUB>(stages, mc, codes_only) + G::kWarps * stages * 8 + kStreamMisc + 1024;
}

// Per-CTA shared-memory budget of the persistent kernel: the measured best
// for 32-row warps; two CTAs per SM for 16-row warps.
constexpr int kHalfSm = 228 * 1024 / 2 - 1024;  // per-CTA budget for two CTAs per SM (1 KB reserved each)
// CTAs per SM the persistent kernel is sized for, and the per-CTA budget.
template <int NSUB>
constexpr int stream_ctas_per_sm() { return Geo<NSUB>::kWarps >= 8 && NSUB == 2 ? 1 : 2; }
template <int NSUB>
constexpr int stream_budget() { return stream_ctas_per_sm<NSUB>() == 1 ? kSmemLimit - 1024 : kHalfSm; }
template <int NSUB>
constexpr int stream_smem_target() {
  return NSUB == 2 && Geo<NSUB>::kWarps == 4 ? W4A16_TC_SMEM_TARGET : stream_budget<NSUB>();
}

// Deepest ring (up to W4A16_TC_MAX_STAGES, at least 2 stages per warp) that
// keeps a CTA's shared memory under the budget.
template <int NSUB>
int stream_stages(int mc, int extra = 0) {
  for (int s = W4A16_TC_MAX_STAGES; s > 2; --s)
    if (stream_smem<NSUB>(s, mc) + extra <= stream_smem_target<NSUB>()) return s;
  return 2;
}

struct DeviceInfo {
  int sms = 152;
  std::set<const void*> attr_done;  // kernels whose shared-memory limit is raised
};

// Raise a kernel's dynamic shared-memory limit once per device.
template <typename Kern>
cudaError_t allow_smem(Kern fn, DeviceInfo& d) {
  const void* key = reinterpret_cast<const void*>(fn);
  if (d.attr_done.count(key)) return cudaSuccess;
  if (cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit)) return e;
  d.attr_done.insert(key);
  return cudaSuccess;
}

// The activations are pre-staged (once per CTA) when the CTA, with a
// two-stage ring per warp, still fits twice on an SM; otherwise every stage
// carries its own activation chunk.  Staging costs each CTA a prologue (copy
// + group sums over all of K); it pays off when every warp has several work
// units to amortise it over.
template <int NSUB>
bool stage_activations(int M, int K, int units, int sms, int extra = 0) {
  return units >= 2 * Geo<NSUB>::kWarps * stream_ctas_per_sm<NSUB>() * sms &&
         stream_smem<NSUB>(2, 0) + xstage_bytes(M, K) + extra <= stream_budget<NSUB>();
}

template <int NSUB>
int staged_stages(int M, int K, int extra = 0) {
  for (int s = W4A16_TC_MAX_STAGES; s > 2; --s)
    if (stream_smem<NSUB>(s, 0) + xstage_bytes(M, K) + extra <= stream_budget<NSUB>()) return s;
  return 2;
}

// Bytes of one per-unit parameter slot with K % 512 != 0: the unit's rows of
// the scales and of the biases (K / 32 bytes a row), each with room for its
// offset modulo 16 and the last stage's reads past the last row (the
// kernel's phalf, twice).
template <int NSUB>
int ptail_slot_bytes(int K) {
  return 2 * ((Geo<NSUB>::kRows * (K / 32) + 45) & ~15);
}

// Shared memory of the persistent kernel with S per-unit parameter slots of
// pslot bytes per warp after everything else: the ring as deep as fits, from
// `stages` down to 2.  Returns the bytes (0 when two stages do not fit) and
// sets stages and par_off.
template <int NSUB>
int unit_param_smem(int& stages, int& par_off, int M, bool staged, int kp, int extra, int pslot, bool codes_only) {
  for (;; --stages) {
    const int smem = stream_smem<NSUB>(stages, staged ? 0 : M, codes_only) + extra + (staged ? xstage_bytes(M, kp) : 0);
    par_off = (smem - 1024 + 15) & ~15;
    const int total = par_off + Geo<NSUB>::kWarps * stages * pslot + 1024;
    if (total <= kSmemLimit) return total;
    if (stages <= 2) return 0;
  }
}

// Launch with, when pdl is set, a programmatic dependency on the previous
// kernel of the stream (the kernels wait for it with griddepcontrol.wait
// before touching anything it may have written), and with clusters of
// `cluster` CTAs along x when cluster > 1.
template <typename Kern, typename... Args>
cudaError_t launch_ex(Kern fn, dim3 grid, dim3 block, int smem, cudaStream_t stream, bool pdl, int cluster,
                      const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, fn, args...);
}

template <int NSUB, bool A, bool X, bool SPLIT, bool ARGMAX = false, bool WHOLEK = false, bool G128 = false,
          bool PT = false>
cudaError_t stream_launch_t(const Maps& map, const StreamParams& p, int sms, int smem, DeviceInfo& d,
                            cudaStream_t stream, bool pdl) {
  constexpr int kW = Geo<NSUB>::kWarps;
  auto* fn = tc_stream_kernel<NSUB, A, X, SPLIT, false, ARGMAX, WHOLEK, G128, PT>;
  if (cudaError_t e = allow_smem(fn, d)) return e;
  int per_sm = 0;
  if (cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kW * 32, smem)) return e;
  if (per_sm < 1) per_sm = 1;
  int grid = sms * per_sm;
  const int need = (p.units + kW - 1) / kW;
  if (grid > need) grid = need;
  return launch_ex(fn, dim3(grid), dim3(kW * 32), smem, stream, pdl, 1, map, p);
}

// Persistent grid for one chunk: every SM filled to its occupancy, never more
// CTAs than there are groups of kWarps work units.  p.tiles / p.units count
// 16 * NSUB-row tiles.  The caller holds g_dev_mu.
template <int NSUB>
cudaError_t launch_stream_t(const Maps& map, StreamParams p, int sms, DeviceInfo& d, cudaStream_t stream, int pdl) {
  const bool allcols = p.M > 1;
  const int extra = p.idx ? kArgmaxSmem : 0;  // the argmax mode's keys
  const int kp = kpad(p.K);
  bool staged = stage_activations<NSUB>(p.M, kp, p.units, sms, extra);
  p.xpitch = staged ? 2 * kp + 64 : 0;
  p.stages = staged ? staged_stages<NSUB>(p.M, kp, extra) : stream_stages<NSUB>(p.M, extra);
  p.prefetch = pdl >= 2;
  int smem = stream_smem<NSUB>(p.stages, staged ? 0 : p.M) + extra;
  if (staged) smem += xstage_bytes(p.M, kp);
  const bool on = pdl > 0;
  using Fn = cudaError_t (*)(const Maps&, const StreamParams&, int, int, DeviceInfo&, cudaStream_t, bool);
  if (p.g128 || p.ptail) {  // whole-K units with their parameter rows in shared memory
    // the ring as deep as fits next to S parameter slots per warp; per-stage
    // activation copies where the pre-staged rows leave no room
    const int pslot = p.g128 ? p.K : ptail_slot_bytes<NSUB>(p.K);
    smem = unit_param_smem<NSUB>(p.stages, p.par_off, p.M, staged, kp, extra, pslot, p.ptail != 0);
    if (!smem && staged) {
      staged = false;
      p.xpitch = 0;
      p.stages = stream_stages<NSUB>(p.M, extra);
      smem = unit_param_smem<NSUB>(p.stages, p.par_off, p.M, false, kp, extra, pslot, p.ptail != 0);
    }
    if (!smem) return cudaErrorInvalidValue;
    if (p.ptail) {  // [allcols][staged][split]: K split over SMs where a workspace is given
      static const Fn pt[2][2][2] = {
          {{stream_launch_t<NSUB, false, false, false, false, false, false, true>,
            stream_launch_t<NSUB, false, false, true, false, false, false, true>},
           {stream_launch_t<NSUB, false, true, false, false, false, false, true>,
            stream_launch_t<NSUB, false, true, true, false, false, false, true>}},
          {{stream_launch_t<NSUB, true, false, false, false, false, false, true>,
            stream_launch_t<NSUB, true, false, true, false, false, false, true>},
           {stream_launch_t<NSUB, true, true, false, false, false, false, true>,
            stream_launch_t<NSUB, true, true, true, false, false, false, true>}}};
      return pt[allcols][staged][p.ks > 1 && p.part != nullptr](map, p, sms, smem, d, stream, on);
    }
    static const Fn g128[2][2] = {{stream_launch_t<NSUB, false, false, false, false, false, true>,
                                   stream_launch_t<NSUB, false, true, false, false, false, true>},
                                  {stream_launch_t<NSUB, true, false, false, false, false, true>,
                                   stream_launch_t<NSUB, true, true, false, false, false, true>}};
    return g128[allcols][staged](map, p, sms, smem, d, stream, on);
  }
  const bool split = p.ks > 1 && p.part != nullptr;
  if (p.ks > 1 && !split) {  // no workspace: whole-K units, the slice sums folded in registers
    static const Fn fold[2][2] = {{stream_launch_t<NSUB, false, false, false, false, true>,
                                   stream_launch_t<NSUB, false, true, false, false, true>},
                                  {stream_launch_t<NSUB, true, false, false, false, true>,
                                   stream_launch_t<NSUB, true, true, false, false, true>}};
    return fold[allcols][staged](map, p, sms, smem, d, stream, on);
  }
  if (p.idx) {  // argmax mode (32-row warps only)
    if (NSUB != 2) return cudaErrorInvalidConfiguration;
    // [allcols][staged][split]
    static const Fn fns[2][2][2] = {
        {{stream_launch_t<2, false, false, false, true>, stream_launch_t<2, false, false, true, true>},
         {stream_launch_t<2, false, true, false, true>, stream_launch_t<2, false, true, true, true>}},
        {{stream_launch_t<2, true, false, false, true>, stream_launch_t<2, true, false, true, true>},
         {stream_launch_t<2, true, true, false, true>, stream_launch_t<2, true, true, true, true>}}};
    return fns[allcols][staged][split](map, p, sms, smem, d, stream, on);
  }
  // [allcols][staged][split]
  static const Fn fns[2][2][2] = {
      {{stream_launch_t<NSUB, false, false, false>, stream_launch_t<NSUB, false, false, true>},
       {stream_launch_t<NSUB, false, true, false>, stream_launch_t<NSUB, false, true, true>}},
      {{stream_launch_t<NSUB, true, false, false>, stream_launch_t<NSUB, true, false, true>},
       {stream_launch_t<NSUB, true, true, false>, stream_launch_t<NSUB, true, true, true>}}};
  return fns[allcols][staged][split](map, p, sms, smem, d, stream, on);
}

// Row subtiles per warp of the persistent kernel for a chunk of M rows.
// 16-row warps fit twice as many per SM; on the shapes the persistent
// kernel serves (LM heads, 16384^2) 32-row warps were measured faster at
// every M, so 16-row warps are used from W4A16_TC_STREAM_NSUB1_MIN_M rows
// on (never, by default).
int stream_nsub(int M) { return M >= W4A16_TC_STREAM_NSUB1_MIN_M ? 1 : 2; }

// Launch shape of the tile kernel for one chunk of M rows.
struct TilePlan {
  int xcap = 0;   // activation rows per x slot
  int R = 1;      // 16-row subtiles per CTA
  int kc = 0;     // CTAs per row tile (cluster size); 0: the tile kernel does not apply
  int nloc = 0;   // stage slots per CTA
  int warps = 0;  // warps per CTA
  int smem = 0;   // dynamic shared memory per CTA
  int ctas = 0;   // grid size (per expert for the routed mode)
};

// CTAs of the tile kernel (80 registers a thread at most) that fit on an SM.
int tile_ctas_per_sm(int warps, int smem) {
  int n = (228 * 1024) / (smem + 1024);
  const int by_regs = 65536 / (warps * 32 * 80);
  const int by_warps = 64 / warps;
  if (by_regs < n) n = by_regs;
  if (by_warps < n) n = by_warps;
  return n < 32 ? n : 32;
}

// The tile kernel serves shapes whose canonical slices are single stages (a
// persistent grid would give each warp about one unit); measured faster
// there at every M even when its CTAs run in several waves, and slower on
// larger shapes.  A tile's slices are dealt to clusters of kc CTAs with at
// most W4A16_TC_TILE_SLICES each; kc grows (up to 8) until a CTA fits in
// shared memory.  `force` drops the size condition.
TilePlan tile_plan_r(const Shape& s, int N, int M, bool force, int R, int ptK = 0) {
  TilePlan tp;
  if (!force && s.nst * s.tiles > W4A16_TC_TILE_MAX_UNITS) return tp;
  const int tiles = cdiv(N, kTile16 * R);
  // Cluster sizes 1, 2, 3, 5 and 8 only: on 2560x10240 and 1536x12288, 5
  // beat 4, 6 and 7 (and 3 beat 4) by 10-40% (measured).
  static const int kSizes[] = {1, 2, 3, 5, 8};
  for (int kc : kSizes) {
    if (kc > s.ks) break;  // a CTA per slice already
    const int ksl = cdiv(s.ks, kc);
    if (ksl > W4A16_TC_TILE_SLICES && kc < kMaxCluster) continue;  // too many slices per CTA
    const int nloc = ksl * s.sl;
    const int smem = tile_smem(nloc, M, s.ks, R, ptK);
    if (smem > kSmemLimit) continue;
    const int warps = R * cdiv(ksl, W4A16_TC_TILE_SLICES_PER_WARP);
    if (warps > kTileMaxWarps) continue;
    tp.xcap = M;
    tp.R = R;
    tp.kc = kc;
    tp.nloc = nloc;
    tp.warps = warps;
    tp.smem = smem;
    tp.ctas = tiles * kc;
    return tp;
  }
  return tp;
}

// With several activation rows, 32-row CTAs (R = 2) halve the activation
// chunks per weight in shared memory; they are taken when they need fewer
// waves of CTAs than 16-row ones (on 2560x10240 at M = 5 the 16-row CTAs no
// longer fit in one wave), or as few when both fit in one (12288x1536 at
// M = 3 / 5: 6.08 -> 5.78 / 6.20 -> 5.98 us; on a tie at two waves 16-row
// CTAs stay faster: 10240x2560 at M = 5, 7.4 against 8.0 us).
// ptK: K when K % 512 != 0 (the padded-K mode's parameter rows), else 0.
TilePlan tile_plan(const Shape& s, int N, int M, bool force, int sms = 152, int ptK = 0) {
  const TilePlan one = tile_plan_r(s, N, M, force, 1, ptK);
  if (M < 2) return one;
  const TilePlan two = tile_plan_r(s, N, M, force, 2, ptK);
  if (two.kc == 0) return one;
  if (one.kc == 0) return two;
  const int w1 = cdiv(one.ctas, sms * tile_ctas_per_sm(one.warps, one.smem));
  const int w2 = cdiv(two.ctas, sms * tile_ctas_per_sm(two.warps, two.smem));
  return (w2 < w1 || (w2 == w1 && w1 == 1)) ? two : one;
}

TileParams tile_params(const Shape& s, const TilePlan& tp, int K, int M, int row0, int* flags, int pdl) {
  TileParams p;
  p.flags = flags;
  p.ids = nullptr;
  p.items = 1;
  p.K = K; p.M = M; p.row0 = row0; p.T = 0; p.E = 1;
  p.nst = s.nst; p.sl = s.sl; p.ks = s.ks;
  p.kc = tp.kc;
  p.nloc = tp.nloc;
  p.xcap = tp.xcap;
  p.prefetch = pdl >= 2;
  return p;
}

// The tile kernel instance for (columns, mode, items, row subtiles).
template <int G>
using TileFn = void (*)(TileArgs<G>, TileParams);
template <int G, bool PT = false>
TileFn<G> tile_fn(bool allcols, bool routed, int R, bool multi = false) {
  if (routed) return tc_tile_kernel<true, true, G, 1, false, PT>;
  if (multi)
    return R == 2 ? tc_tile_kernel<true, false, G, 2, true, PT> : tc_tile_kernel<true, false, G, 1, true, PT>;
  if (R == 2) return allcols ? tc_tile_kernel<true, false, G, 2, false, PT> : tc_tile_kernel<false, false, G, 2, false, PT>;
  return allcols ? tc_tile_kernel<true, false, G, 1, false, PT> : tc_tile_kernel<false, false, G, 1, false, PT>;
}

// K % 512 != 0 (a plan made with ptK = K): the padded-K instances, whose
// parameter rows come by bulk copy (no tensor map for them).
cudaError_t launch_tile(const LaunchArgs& a, const Shape& s, const TilePlan& tp, DeviceInfo& d, bool routed) {
  TileArgs<1> ta;
  const bool pt = a.K % kStageK != 0;
  const int64_t rows = routed ? (int64_t)a.N * a.E : a.N;
  if (pt) {
    if (cudaError_t e = make_code_map(&ta.maps[0].codes, a.Wq, rows, a.K, kTile16 * tp.R)) return e;
    ta.maps[0].scales = ta.maps[0].codes;  // unused
    ta.maps[0].biases = ta.maps[0].codes;
  } else if (cudaError_t e = make_maps(&ta.maps[0], a.Wq, a.S, a.B, rows, a.K, kTile16 * tp.R)) {
    return e;
  }
  ta.S[0] = a.S;
  ta.B[0] = a.B;
  ta.x[0] = a.x;
  ta.y[0] = a.y;
  ta.N[0] = a.N;
  ta.tile0[0] = 0;
  ta.tile0[1] = cdiv(a.N, kTile16 * tp.R);
  TileParams p = tile_params(s, tp, a.K, a.M, a.row0, a.flags, a.pdl);
  if (routed) {
    p.ids = a.ids;
    p.T = a.T;
    p.E = a.E;
    p.prefetch = 0;  // the weights to read depend on the ids
  }
  TileFn<1> fn = pt ? tile_fn<1, true>(a.M > 1, routed, tp.R, !routed && a.M > tp.xcap)
                    : tile_fn<1>(a.M > 1, routed, tp.R, !routed && a.M > tp.xcap);
  if (cudaError_t e = allow_smem(fn, d)) return e;
  const dim3 grid(tp.ctas, routed ? a.E : 1);
  return launch_ex(fn, grid, dim3(tp.warps * 32), tp.smem, a.stream, a.pdl > 0, tp.kc, ta, p);
}

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
//   [kWsTiles] int counters (zero between launches: tile arrivals, and the
//   last two for the unit scheduler) | fp32 slice partials [units][8][rows]
//   (rows = 16 or 32 per unit).
// ksplit > 1 only happens when a chunk has fewer than kTargetUnits 32-row
// tiles, and then (from the slicing rule of tc_shape) it has fewer than
// 2 kTargetUnits 32-row units: twice as many 16-row ones, the same bytes.
// One fixed-size buffer serves every shape and never needs to grow; the
// launch checks it all the same.
constexpr int kWsTiles = 8192;
constexpr size_t kWsCounterBytes = (size_t)kWsTiles * 4;
constexpr size_t kWsPartBytes = (size_t)2 * kTargetUnits * 8 * 32 * 4;
constexpr size_t kWsBytes = kWsCounterBytes + kWsPartBytes;

// Work decomposition of the persistent kernel for a chunk of M rows.
struct StreamWork {
  int nsub, rows, tiles, units;
};

StreamWork stream_work(const Shape& s, int N, int M) {
  StreamWork w;
  w.nsub = stream_nsub(M);
  w.rows = 16 * w.nsub;
  w.tiles = cdiv(N, w.rows);
  w.units = w.tiles * s.ks;
  return w;
}

// The last 32 counters of the workspace belong to the persistent kernel's
// schedulers: the unit-grab counter, the argmax mode's finished-CTA counter
// and its eight 64-bit keys; the tiles' arrival counters are the others.
constexpr int kWsSched = kWsTiles - 2;   // grab counter, then the finished-CTA counter
constexpr int kWsBest = kWsTiles - 32;   // u64 [8] (byte offset a multiple of 8)

bool workspace_fits(const Shape& s, const StreamWork& w) {
  return s.ks == 1 || (w.tiles <= kWsBest && (size_t)w.units * 8 * w.rows * 4 <= kWsPartBytes);
}

cudaError_t launch_stream(const Maps& maps, StreamParams p, const StreamWork& w, DeviceInfo& d,
                          cudaStream_t stream, int pdl) {
  p.tiles = w.tiles;
  p.units = p.ks > 1 && (!p.part || p.g128) ? w.tiles : w.units;  // whole-K units
  p.kfull = p.nst % p.sl == 0 ? p.ks : p.ks - 1;
#if W4A16_TC_STREAM_NSUB1_MIN_M <= 8  // else no chunk (8 rows at most) takes 16-row warps
  if (w.nsub == 1) return launch_stream_t<1>(maps, p, d.sms, d, stream, pdl);
#endif
  return launch_stream_t<2>(maps, p, d.sms, d, stream, pdl);
}

// Point the persistent kernel's counters, partials and argmax keys into a
// caller's workspace of kWsBytes.
void use_workspace(StreamParams& p, void* ws) {
  p.cnt = static_cast<int*>(ws);
  p.sched = p.cnt + kWsSched;
  p.done = p.cnt + kWsSched + 1;
  p.best = reinterpret_cast<unsigned long long*>(p.cnt + kWsBest);
  p.part = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsCounterBytes);
}

}  // namespace

size_t tc_workspace_bytes() { return kWsBytes; }

cudaError_t encode_map_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, int64_t inner,
                          int64_t outer, int64_t row_bytes, int box_inner, int box_outer, CUtensorMapSwizzle swizzle) {
  if (cudaError_t e = get_encoder()) return e;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, type, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// K % 512 != 0: the persistent kernel's per-unit parameter slots fit next to
// a two-stage ring with per-stage copies of eight activation rows (the most
// shared memory any chunk takes).
bool tc_ptail_fits(int K) {
  int stages = 2, par_off = 0;
  return unit_param_smem<2>(stages, par_off, kMaxChunk, false, kpad(K), 0, ptail_slot_bytes<2>(K), true) > 0;
}

bool tc_supported(int N, int K) {
  (void)N;
  if (K <= 0 || K % kGroup) return false;
  return K % kStageK == 0 || tc_ptail_fits(K);  // K % 512 != 0 runs padded to whole stages
}

bool tc_tile_fits(int N, int K, int M) {
  return tile_plan(tc_shape(N, K), N, M, true, 152, K % kStageK ? K : 0).kc > 0;
}

void plan_tc(int N, int K, int tc_path, w4a16_plan* p) {
  const Shape s = tc_shape(N, K);
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    sms = device_info(dev).sms;
  } else {
    cudaGetLastError();
  }
  p->ksplit = s.ks;
  p->slice_k = s.sl * kStageK;
  p->rows_per_tile = kTileRows;
  p->units = s.units;
  p->kernel = tc_path == 1 ? W4A16_KERNEL_TC_STREAM : tc_path == 2 ? W4A16_KERNEL_TC_TILE : W4A16_KERNEL_TC;
  const int ptK = K % kStageK ? K : 0;
  if (ptK && tc_path != 1) {  // the tile kernel where it applies (one row, with a workspace)
    const TilePlan tp = tile_plan(s, N, 1, tc_path == 2, sms, ptK);
    if (tp.kc > 0) {
      p->rows_per_tile = kTile16;
      p->threads = tp.warps * 32;
      p->grid_x = tp.ctas;
      p->smem_bytes = tp.smem;
      p->workspace_bytes = 0;
      return;
    }
  }
  if (ptK) {  // the persistent kernel, parameter rows per unit
    const StreamWork w = stream_work(s, N, 1);
    const int kp = kpad(K), pslot = ptail_slot_bytes<2>(K);
    bool staged = stage_activations<2>(1, kp, w.tiles, sms);
    int stages = staged ? staged_stages<2>(1, kp) : stream_stages<2>(1), par_off = 0;
    int smem = unit_param_smem<2>(stages, par_off, 1, staged, kp, 0, pslot, true);
    if (!smem && staged) {
      stages = stream_stages<2>(1);
      smem = unit_param_smem<2>(stages, par_off, 1, false, kp, 0, pslot, true);
    }
    const int per_sm = smem > 0 && kSmemLimit / smem > 0 ? kSmemLimit / smem : 1;
    const int need = cdiv(w.units, Geo<2>::kWarps);
    p->rows_per_tile = w.rows;
    p->units = w.units;  // split over SMs with a workspace (whole-K units without)
    p->threads = Geo<2>::kWarps * 32;
    p->grid_x = sms * per_sm < need ? sms * per_sm : need;
    p->smem_bytes = smem;
    p->workspace_bytes = s.ks > 1 ? (int)kWsBytes : 0;
    return;
  }
  const TilePlan tp = tc_path == 1 ? TilePlan() : tile_plan(s, N, 1, tc_path == 2);
  p->workspace_bytes = 0;
  if (tp.kc > 0) {  // clusters of kc CTAs per 16-row tile
    p->rows_per_tile = kTile16;
    p->threads = tp.warps * 32;
    p->grid_x = tp.ctas;
    p->smem_bytes = tp.smem;
    return;
  }
  p->workspace_bytes = (int)kWsBytes;
  const StreamWork w = stream_work(s, N, 1);
  int smem, warps;
  if (w.nsub == 1) {
    const bool staged = stage_activations<1>(1, kpad(K), w.units, sms);
    smem = staged ? stream_smem<1>(staged_stages<1>(1, kpad(K)), 0) + xstage_bytes(1, kpad(K))
                  : stream_smem<1>(stream_stages<1>(1), 1);
    warps = Geo<1>::kWarps;
  } else {
    const bool staged = stage_activations<2>(1, kpad(K), w.units, sms);
    smem = staged ? stream_smem<2>(staged_stages<2>(1, kpad(K)), 0) + xstage_bytes(1, kpad(K))
                  : stream_smem<2>(stream_stages<2>(1), 1);
    warps = Geo<2>::kWarps;
  }
  const int per_sm = kSmemLimit / smem > 0 ? kSmemLimit / smem : 1;
  int grid = sms * per_sm;
  const int need = (w.units + warps - 1) / warps;
  if (grid > need) grid = need;
  p->rows_per_tile = w.rows;
  p->units = w.units;
  p->threads = warps * 32;
  p->grid_x = grid;
  p->smem_bytes = smem;
}

cudaError_t launch_tc_ptail(const LaunchArgs& a);

// w4a16_mm (idx == nullptr) or, always on the persistent kernel, its argmax
// mode (w4a16_mm_argmax).
cudaError_t launch_tc_impl(const LaunchArgs& a, int32_t* idx, uint16_t* val) {
  const Shape s = tc_shape(a.N, a.K);
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  StreamParams p{};
  p.x = a.x; p.S = a.S; p.B = a.B; p.y = a.y; p.flags = a.flags;
  p.idx = idx; p.val = val;
  p.N = a.N; p.K = a.K; p.M = a.M; p.row0 = a.row0;
  p.nst = s.nst; p.sl = s.sl; p.ks = s.ks; p.tiles = s.tiles; p.units = s.units;
  p.stages = 2;
  p.xpitch = 0;
  p.part = nullptr;
  p.cnt = nullptr;
  p.sched = nullptr;
  if (a.K % kStageK) {  // parameter rows by bulk copy: no argmax mode or prefill kernel
    if (idx || a.tc_path == 3) return cudaErrorInvalidConfiguration;
    if (a.tc_path != 1) {
      // the tile kernel where it applies (as below; without a workspace the
      // persistent grid's units would be whole-K, so clusters hold split shapes)
      std::lock_guard<std::mutex> lk(g_dev_mu);
      DeviceInfo& d = device_info(dev);
      const bool have_ws = a.ws != nullptr && a.ws_bytes >= kWsBytes;
      const int mc = min(a.M, kMaxChunk);
      TilePlan tp = tile_plan(s, a.N, mc, a.tc_path == 2, d.sms, a.K);
      if (tp.kc == 0 && a.tc_path != 2 && (s.ks > 1 && !have_ws)) tp = tile_plan(s, a.N, mc, true, d.sms, a.K);
      if (tp.kc > 0) return launch_tile(a, s, tp, d, false);
      if (a.tc_path == 2) return cudaErrorInvalidConfiguration;
    }
    return launch_tc_ptail(a);  // takes g_dev_mu itself
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = device_info(dev);
  const bool have_ws = a.ws != nullptr && a.ws_bytes >= kWsBytes;
  if (idx && !have_ws) return cudaErrorInvalidValue;  // the argmax mode merges its keys in the workspace
  // Many rows: the tcgen05 kernel expands each weight once for all of them
  if (!idx && (a.tc_path == 3 || (a.tc_path == 0 && a.M >= kPrefillMinM))) return launch_prefill(a, s.sl * kStageK);
  if (a.tc_path != 1 && !idx) {
    // one launch for all M rows: eight at a time over the resident weights
    const TilePlan tp = tile_plan(s, a.N, min(a.M, kMaxChunk), a.tc_path == 2, d.sms);
    if (tp.kc > 0) return launch_tile(a, s, tp, d, false);
    if (a.tc_path == 2) return cudaErrorInvalidConfiguration;
    // K split over SMs needs the workspace; without one, the tile kernel's
    // clusters add the slice sums in distributed shared memory where a
    // cluster can hold a tile's K range
    if (s.ks > 1 && !have_ws) {
      const TilePlan tf = tile_plan(s, a.N, min(a.M, kMaxChunk), true, d.sms);
      if (tf.kc > 0) return launch_tile(a, s, tf, d, false);
    }
  }
  // Persistent kernel.  With a workspace: units dealt over the whole grid
  // from its counter, K split over SMs through its partials.  Without:
  // units dealt inside each CTA, and a split K taken by whole-K units that
  // fold the slice sums in registers (the same canonical sums).
  if (have_ws) use_workspace(p, a.ws);
  if (a.fault_wait) {  // debug: one stage's wait runs out after 4096 tries
    p.fault_tx = 16;
    p.wait_limit = 1u << 12;
  }
  // the persistent kernel: one launch per chunk of at most eight rows
  for (int r0 = 0; r0 < a.M; r0 += kMaxChunk) {
    p.row0 = a.row0 + r0;
    p.M = min(kMaxChunk, a.M - r0);
    const StreamWork w = stream_work(s, a.N, p.M);
    Maps maps;
    if (cudaError_t e = make_maps(&maps, a.Wq, a.S, a.B, a.N, a.K, w.rows)) return e;
    if (p.part && !workspace_fits(s, w)) return cudaErrorInvalidValue;
    if (cudaError_t e = launch_stream(maps, p, w, d, a.stream, a.pdl)) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_tc(const LaunchArgs& a, const w4a16_plan& plan) {
  (void)plan;
  return launch_tc_impl(a, nullptr, nullptr);
}

cudaError_t launch_tc_argmax(const LaunchArgs& a, int32_t* idx, uint16_t* val) {
  return idx ? launch_tc_impl(a, idx, val) : cudaErrorInvalidValue;
}

// Tokens per chunk of the routed tile kernel: twice the mean per expert (at
// least one, at most eight); an expert with more tokens takes more chunks
// over the same resident weights.
int routed_xcap(int T, int E) {
  int x = 2 * cdiv(T, E);
  if (x > T) x = T;
  if (x > kMaxChunk) x = kMaxChunk;
  return x < 1 ? 1 : x;
}

// The persistent kernel in routed mode (T <= kRoutedStreamMaxT): 32-row
// whole-K units of the chunks the ids select, dealt round-robin over a full
// grid.  Nothing is requested before the wait for earlier kernels (the ids
// decide which weights are read).  The caller holds g_dev_mu.
cudaError_t launch_stream_routed(const LaunchArgs& a, DeviceInfo& d) {
  const Shape s = tc_shape(a.N, a.K);
  StreamParams p{};
  p.x = a.x; p.S = a.S; p.B = a.B; p.y = a.y; p.flags = a.flags;
  p.N = a.N; p.K = a.K; p.M = routed_xcap(a.T, a.E); p.row0 = 0;
  p.nst = s.nst; p.sl = s.sl; p.ks = s.ks;
  p.tiles = cdiv(a.N, kTileRows);
  p.stages = stream_stages<2>(p.M);
  p.ids = a.ids; p.T = a.T; p.E = a.E;
  p.ptail = a.K % kStageK != 0;
  // Before the ids arrive, pull the first stage of every expert into L2 when
  // that costs at most 16 MB (the budget of bytes read on speculation).
  p.l2_stages = !p.ptail && a.pdl >= 2 &&
                (int64_t)a.E * a.N * (kStageK / 2 + kStageK / kGroup * 4) <= (16 << 20) ? 1 : 0;
  Maps maps;
  if (p.ptail) {  // K % 512 != 0: the parameter rows come per unit by bulk copy
    if (cudaError_t e = make_code_map(&maps.codes, a.Wq, (int64_t)a.N * a.E, a.K, kTileRows)) return e;
    maps.scales = maps.codes;
    maps.biases = maps.codes;
  } else if (cudaError_t e = make_maps(&maps, a.Wq, a.S, a.B, (int64_t)a.N * a.E, a.K, kTileRows)) {
    return e;
  }
  int smem = stream_smem<2>(p.stages, p.M, p.ptail != 0) + routed_table_bytes(a.T);
  if (p.ptail) {
    const int pslot = ptail_slot_bytes<2>(a.K);
    for (;; --p.stages) {
      smem = stream_smem<2>(p.stages, p.M, true) + routed_table_bytes(a.T);
      p.par_off = (smem - 1024 + 15) & ~15;
      smem = p.par_off + Geo<2>::kWarps * p.stages * pslot + 1024;
      if (smem <= kSmemLimit) break;
      if (p.stages <= 2) return cudaErrorInvalidValue;
    }
  }
  constexpr int kW = Geo<2>::kWarps;
  auto* fn = p.ptail ? (p.M > 1 ? tc_stream_kernel<2, true, false, false, true, false, false, false, true>
                                : tc_stream_kernel<2, false, false, false, true, false, false, false, true>)
                     : (p.M > 1 ? tc_stream_kernel<2, true, false, false, true>
                                : tc_stream_kernel<2, false, false, false, true>);
  if (cudaError_t e = allow_smem(fn, d)) return e;
  int per_sm = 0;
  if (cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kW * 32, smem)) return e;
  if (per_sm < 1) per_sm = 1;
  int grid = d.sms * per_sm;
  const int need = cdiv(a.T * p.tiles, kW);  // at most T chunks
  if (grid > need) grid = need;
  return launch_ex(fn, dim3(grid), dim3(kW * 32), smem, a.stream, a.pdl > 0, 1, maps, p);
}

cudaError_t launch_tc_id(const LaunchArgs& a, const w4a16_plan& plan) {
  (void)plan;
  const Shape s = tc_shape(a.N, a.K);
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  if (a.K % kStageK) {
    // whole-K units with per-unit parameter rows: the persistent routed mode
    // only, kRoutedStreamMaxT tokens per launch (rows are independent)
    if (a.tc_path == 2) return cudaErrorInvalidConfiguration;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = device_info(dev);
    for (int t0 = 0; t0 < a.T; t0 += kRoutedStreamMaxT) {
      LaunchArgs b = a;
      b.T = min(kRoutedStreamMaxT, a.T - t0);
      b.ids = a.ids + t0;
      b.x = a.x + (int64_t)t0 * a.K;
      b.y = a.y + (int64_t)t0 * a.N;
      if (cudaError_t e = launch_stream_routed(b, d)) return e;
    }
    return cudaSuccess;
  }
  if (a.tc_path != 2 && a.T <= kRoutedStreamMaxT) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = device_info(dev);
    // The persistent routed mode pays when the chunks can give every warp of
    // its grid (two CTAs of four warps per SM) a unit: at most T chunks of
    // ceil(N / 32) units each.  With fewer, the tile kernel splits K over
    // more CTAs instead (measured: 8 x 6144x2048 at T = 8: 12.6 against 15.2
    // us; 8 x 2048x2048 at T = 8: 11.2 against 7.5; 16 x 512x8192 at T = 4:
    // 26.1 against 7.5).
    if (a.tc_path == 1 || (int64_t)a.T * cdiv(a.N, kTileRows) >= 8 * d.sms) return launch_stream_routed(a, d);
  }
  if (a.tc_path != 1) {  // the tile kernel in routed mode, where it fits
    const TilePlan tp = tile_plan_r(s, a.N, routed_xcap(a.T, a.E), true, 1);
    if (tp.kc > 0) {
      std::lock_guard<std::mutex> lk(g_dev_mu);
      return launch_tile(a, s, tp, device_info(dev), true);
    }
  }
  RoutedParams p;
  p.x = a.x; p.S = a.S; p.B = a.B; p.y = a.y; p.ids = a.ids; p.flags = a.flags;
  p.N = a.N; p.K = a.K; p.T = a.T; p.E = a.E;
  p.nst = s.nst; p.sl = s.sl; p.ks = s.ks;
  p.warps = s.ks < kRoutedWarps ? s.ks : kRoutedWarps;
  p.xcap = a.T < kMaxChunk ? a.T : kMaxChunk;  // a chunk never holds more tokens than there are
  // a ring no deeper than the stages a warp has (all in flight at once), at most 3
  const int per_warp = (s.ks + p.warps - 1) / p.warps * s.sl;
  p.stages = per_warp < 3 ? per_warp : 3;
  while (p.stages > 1 && routed_smem(p.warps, p.stages, p.ks, p.xcap) > kSmemLimit) --p.stages;
  while (p.warps > 1 && routed_smem(p.warps, p.stages, p.ks, p.xcap) > kSmemLimit) --p.warps;
  const int smem = routed_smem(p.warps, p.stages, p.ks, p.xcap);
  if (smem > kSmemLimit) return cudaErrorInvalidConfiguration;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = device_info(dev);
    if (cudaError_t e = allow_smem(tc_routed_kernel, d)) return e;
  }
  Maps maps;
  if (cudaError_t e = make_maps(&maps, a.Wq, a.S, a.B, (int64_t)a.N * a.E, a.K)) return e;
  return launch_ex(tc_routed_kernel, dim3(s.tiles, a.E), dim3(p.warps * 32), smem, a.stream, a.pdl > 0, 1, maps, p);
}

bool tc_group_supported(const int* N, int count, int K) {
  if (count < 1 || count > kMaxGroup || K % kStageK) return false;
  for (int i = 0; i < count; ++i) {
    const Shape s = tc_shape(N[i], K);
    if (s.nst * s.tiles > W4A16_TC_TILE_MAX_UNITS) return false;  // each item alone would take the tile kernel
  }
  return tile_plan(tc_shape(N[0], K), N[0], kMaxChunk, false).kc > 0;
}

// One tile-kernel launch over items that share K and M: their tiles follow
// one another in the grid; every item keeps its own canonical slicing (a
// function of K alone for these shapes), so its rows equal a w4a16_mm call
// on it bit for bit.
cudaError_t launch_tc_group(const GroupItem* items, int count, int M, int row0, int K, int pdl, int* flags,
                            cudaStream_t stream) {
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  const Shape s = tc_shape(items[0].N, K);
  int Ntot = 0;
  for (int i = 0; i < count; ++i) Ntot += cdiv(items[i].N, 32) * 32;
  const TilePlan tp = tile_plan(s, Ntot, min(M, kMaxChunk), false);  // depends on N only through the CTA count
  if (tp.kc == 0) return cudaErrorInvalidConfiguration;
  const int rows = kTile16 * tp.R;
  TileArgs<kMaxGroup> ta;
  int tiles = 0;
  for (int i = 0; i < count; ++i) {
    if (cudaError_t e = make_maps(&ta.maps[i], items[i].Wq, items[i].S, items[i].B, items[i].N, K, rows)) return e;
    ta.S[i] = items[i].S;
    ta.B[i] = items[i].B;
    ta.x[i] = items[i].x;
    ta.y[i] = items[i].y;
    ta.N[i] = items[i].N;
    ta.tile0[i] = tiles;
    tiles += cdiv(items[i].N, rows);
  }
  for (int i = count; i < kMaxGroup; ++i) {
    ta.maps[i] = ta.maps[0];
    ta.S[i] = nullptr;
    ta.B[i] = nullptr;
    ta.x[i] = nullptr;
    ta.y[i] = nullptr;
    ta.N[i] = 0;
    ta.tile0[i] = tiles;
  }
  ta.tile0[kMaxGroup] = tiles;
  TileParams p = tile_params(s, tp, K, M, row0, flags, pdl);
  p.items = count;
  TileFn<kMaxGroup> fn = tile_fn<kMaxGroup>(M > 1, false, tp.R, M > tp.xcap);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = device_info(dev);
  if (cudaError_t e = allow_smem(fn, d)) return e;
  return launch_ex(fn, dim3(tiles * tp.kc), dim3(tp.warps * 32), tp.smem, stream, pdl > 0, tp.kc, ta, p);
}

// ---- group-128 tables ---------------------------------------------------------------------
//
// Scales and biases with one pair per 128 codes ([N][K/128], the tiny-llm
// book's layout), read natively: the persistent grid in whole-K units, each
// unit's parameter rows brought into shared memory by one bulk copy per
// table with the unit's first stage (the rows are K / 64 bytes apart, too
// irregular for a tensor map).  Every 64-group is rescaled with its
// 128-group's pair, so the results equal the group-64 kernels on the
// expanded tables bit for bit.  Rows eight at a time, one launch per chunk.
cudaError_t launch_tc_g128(const LaunchArgs& a) {
  const Shape s = tc_shape(a.N, a.K);
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  StreamParams p{};
  p.x = a.x; p.S = a.S; p.B = a.B; p.y = a.y; p.flags = a.flags;
  p.N = a.N; p.K = a.K;
  p.nst = s.nst; p.sl = s.sl; p.ks = s.ks;
  p.stages = 2;
  p.g128 = 1;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = device_info(dev);
  if (a.ws != nullptr && a.ws_bytes >= kWsBytes) {  // the grid-wide unit counter; no K split
    use_workspace(p, a.ws);
    p.part = nullptr;
  }
  for (int r0 = 0; r0 < a.M; r0 += kMaxChunk) {
    p.row0 = a.row0 + r0;
    p.M = min(kMaxChunk, a.M - r0);
    const StreamWork w = stream_work(s, a.N, p.M);
    if (w.nsub != 2) return cudaErrorInvalidConfiguration;
    Maps maps;
    if (cudaError_t e = make_code_map(&maps.codes, a.Wq, a.N, a.K, w.rows)) return e;
    maps.scales = maps.codes;  // unused: the parameters come by bulk copy
    maps.biases = maps.codes;
    if (cudaError_t e = launch_stream(maps, p, w, d, a.stream, a.pdl)) return e;
  }
  return cudaSuccess;
}

// K % 512 != 0: the persistent grid over K padded to whole stages (the
// canonical slicing of the padded K).  No tensor map takes parameter rows
// K / 32 bytes apart, so each unit's rows of the scales and biases (over the
// whole K) come by bulk copy with its first stage, as for group-128 tables.
// With a workspace and one activation row the K split goes over SMs through
// it as for K % 512 == 0 (9216x2304: 12.4 -> 10.9 us); otherwise the units
// are whole-K, the slice sums folded in registers (with more rows the split
// launch's staged activations and parameter slots leave room for one CTA per
// SM: 9216x2304 at M = 5 19.3 us split against 12.3 whole-K).  Rows eight at
// a time, one launch per chunk.
cudaError_t launch_tc_ptail(const LaunchArgs& a) {
  const Shape s = tc_shape(a.N, a.K);
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  StreamParams p{};
  p.x = a.x; p.S = a.S; p.B = a.B; p.y = a.y; p.flags = a.flags;
  p.N = a.N; p.K = a.K;
  p.nst = s.nst; p.sl = s.sl; p.ks = s.ks;
  p.stages = 2;
  p.ptail = 1;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = device_info(dev);
  if (a.ws != nullptr && a.ws_bytes >= kWsBytes) use_workspace(p, a.ws);
  float* const part = p.part;
  for (int r0 = 0; r0 < a.M; r0 += kMaxChunk) {
    p.row0 = a.row0 + r0;
    p.M = min(kMaxChunk, a.M - r0);
    const StreamWork w = stream_work(s, a.N, p.M);
    if (w.nsub != 2) return cudaErrorInvalidConfiguration;
    p.part = p.M == 1 && workspace_fits(s, w) ? part : nullptr;
    Maps maps;
    if (cudaError_t e = make_code_map(&maps.codes, a.Wq, a.N, a.K, w.rows)) return e;
    maps.scales = maps.codes;  // unused: the parameters come by bulk copy
    maps.biases = maps.codes;
    if (cudaError_t e = launch_stream(maps, p, w, d, a.stream, a.pdl)) return e;
  }
  return cudaSuccess;
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
  if (K % kStageK) return tc_ptail_fits(K);  // whole-K units: no scratch
  const Shape s = tc_shape(N, K);
  for (int M = 1; M <= kMaxChunk; ++M)
    if (!workspace_fits(s, stream_work(s, N, M))) return false;
  return true;
}

cudaError_t launch_tc_noalloc(const LaunchArgs& a) {
  if (a.K % kStageK) return launch_tc_ptail(a);  // a.ws is null: units dealt inside each CTA
  const Shape s = tc_shape(a.N, a.K);
  const StreamWork w = stream_work(s, a.N, a.M);
  if (!workspace_fits(s, w)) return cudaErrorInvalidValue;
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  StreamParams p{};
  p.x = a.x; p.S = a.S; p.B = a.B; p.y = a.y; p.flags = a.flags;
  p.N = a.N; p.K = a.K; p.M = a.M; p.row0 = a.row0;
  p.nst = s.nst; p.sl = s.sl; p.ks = s.ks; p.tiles = s.tiles; p.units = s.units;
  p.stages = 2;
  p.xpitch = 0;
  p.part = nullptr;
  p.cnt = nullptr;
  p.sched = nullptr;
  Maps maps;
  if (cudaError_t e = make_maps(&maps, a.Wq, a.S, a.B, a.N, a.K, w.rows)) return e;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = device_info(dev);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaError_t e = cudaGetSymbolAddress((void**)&ptr, g_noalloc_scratch)) return e;
    g_noalloc_ptr[dev] = ptr;
  }
  p.cnt = static_cast<int*>(g_noalloc_ptr[dev]);
  p.sched = p.cnt + kWsSched;
  p.part = reinterpret_cast<float*>(static_cast<char*>(g_noalloc_ptr[dev]) + kWsCounterBytes);
  // The array keeps whatever the previous call left: the counters must start
  // at zero (every launch also leaves them at zero when it completes).
  if (s.ks > 1)
    if (cudaError_t e = cudaMemsetAsync(p.cnt, 0, (size_t)w.tiles * 4, a.stream)) return e;
  if (cudaError_t e = cudaMemsetAsync(p.sched, 0, 2 * sizeof(int), a.stream)) return e;
  return launch_stream(maps, p, w, d, a.stream, a.pdl);
}

}  // namespace w4a16

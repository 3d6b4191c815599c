/*
 * stq1.h -- C ABI of the STQ1_0 ternary matmul in libw4a16.so (sm_103a).
 *
 * Citation (page title; sections in quotes):
 *   [HY4] "Hy4-preview Metal kernels for llama.cpp"
 *
 * The format ([HY4 "Notes and gotchas"], the block-layout and 42-byte-stride
 * notes).  A row of K weights is K/256 blocks of 42 bytes:
 *   bytes  0..31  qs:   64 four-bit group codes, group g in byte g/2, low
 *                       nibble for even g
 *   bytes 32..39  sign: 64 group sign bits, group g at bit g%8 of byte 32+g/8
 *   bytes 40..41  d:    fp16 scale, little endian
 * Weight w (0..255) of a block is lane p = (w%64)/16 of group
 * g = (w/64)*16 + w%16.  A group's four lanes ([HY4 "Results", the fourth
 * decode pass]): the code's high two bits name the zero lane; of the other
 * three lanes, taken in ascending order, bit 0 negates the first and bit 1
 * the second (the page does not say which two lanes the flips reach; this is
 * the reading taken); the group's sign bit negates all four.  A weight is
 * d * v with v in {-1, 0, +1}.
 *
 * The operation (the page's kernel table: kernel_mul_mv_stq1_0_f32 for one
 * row, _ext_ for 2..8 rows, mul_mv_id / mul_mm_id for routed experts,
 * get_rows for the row gather):
 *   y[m][n] = sum_k x[m][k] * W[n][k]            float32 x and y
 *
 * Precision.  Per group the four activations enter as a signed sum
 * (x_r + e_q x_q) + e_p x_p over the three nonzero lanes p < q < r, rounded
 * to float32 after each addition; the 64 group sums of a block are added in
 * four chains (groups g = i mod 4, in order) and then (s0 + s1) + (s2 + s3);
 * y += d * block_sum with a fused multiply-add per block; the K slices are
 * added in slice order.  Bound (the parity tests use it):
 *   |y - y_ref| <= (2^-16 + (K/256 + 16) * 2^-23) * sum_k |x[m][k] W[n][k]|
 * Non-finite activations give non-finite outputs.
 *
 * Batch invariance.  The K split and every reduction order depend on (N, K)
 * only; row m of any call equals, bit for bit, the one-row call on x[m], and
 * stq1_mm_id rows equal stq1_mm on the selected expert.
 *
 * Device layout.  The compute calls read a repacked copy (stq1_pack): for
 * every 16-row tile and block a 672-byte record (16 rows x 42 bytes, the
 * same bytes) in which each row's codes, sign bits and scale are
 * contiguous, for a kernel that gives every lane one row:
 *   bytes   0..255  qs bytes 0..15 of row r at 16*r
 *   bytes 256..511  qs bytes 16..31 of row r at 256 + 16*r
 *   bytes 512..639  sign bytes 0..7 of row r at 512 + 8*r
 *   bytes 640..671  d of row r at 640 + 2*r
 * Records are ordered [ceil(N/16)][K/256]; rows past N are zero.
 *
 * Ownership and synchronisation.  All tensor pointers are DEVICE pointers
 * owned by the caller; `stream` is a cudaStream_t (NULL = legacy default
 * stream).  Calls only enqueue work and never synchronise.  None allocates.
 *
 * Errors: a w4a16_status (include/w4a16.h) and w4a16_last_error().
 * Arguments are checked on the host before any launch; a rejected call
 * writes nothing.  An expert or row id out of range gives a zero output row
 * and raises the device flag read by w4a16_device_status.
 */
#ifndef STQ1_H
#define STQ1_H

#include <stddef.h>
#include <stdint.h>

#include "w4a16.h"

#ifdef __cplusplus
extern "C" {
#endif

#define STQ1_BLOCK_WEIGHTS 256
#define STQ1_BLOCK_BYTES 42
#define STQ1_TILE_ROWS 16
#define STQ1_RECORD_BYTES 672
#define STQ1_MAX_K 32768

/* Bytes of the repacked copy of an N x K matrix: ceil(N/16) * (K/256) * 672,
 * or 0 when N < 1, K < 256, K > STQ1_MAX_K or K % 256 != 0. */
size_t stq1_packed_bytes(int N, int K);

/* Repack blocks[N][K/256][42] (the page's layout; 2-byte aligned, the
 * page's "42-byte block stride" note) into `packed` (16-byte aligned,
 * stq1_packed_bytes(N, K) bytes). */
int stq1_pack(const uint8_t* blocks, uint8_t* packed, int N, int K, void* stream);

/* y[M][N] = x[M][K] W^T with W given as its repacked copy.  x 16-byte
 * aligned, y 4-byte aligned; M >= 0 (M = 0 is a no-op); rows go through in
 * passes of at most rows_per_pass (stq1_get_plan, 8), each a single launch. */
int stq1_mm(const float* x, const uint8_t* packed, float* y, int M, int N, int K, void* stream);

/* Routed experts: packed holds E repacked N x K matrices back to back
 * (stride stq1_packed_bytes(N, K)); y[t] = W[ids[t]] x[t] for T tokens, one
 * expert id each.  One launch; each expert's tokens are gathered on the GPU. */
int stq1_mm_id(const float* x, const uint8_t* packed, const int32_t* ids, float* y, int T, int N, int K, int E,
               void* stream);

/* Row gather: out[t][k] = W[ids[t]][k] as float32 (exact: d * v). */
int stq1_get_rows(const uint8_t* packed, const int32_t* ids, float* out, int T, int N, int K, void* stream);

/* The launch plan of (N, K): 256 weight rows per CTA, K split into ksplit
 * slices (the CTAs of one cluster, at most 8) of blocks_per_slice blocks
 * (the last may be shorter), at most rows_per_pass activation rows per
 * launch. */
typedef struct {
  int ksplit;
  int blocks_per_slice;
  int rows_per_pass;
} stq1_plan;

int stq1_get_plan(int N, int K, stq1_plan* out);

#ifdef __cplusplus
}
#endif

#endif /* STQ1_H */

/*
 * w4a16_synth.h -- seeded, counter-based generator for synthetic W4A16 inputs.
 *
 * This library makes the inputs that both the CUDA path and the CPU oracle
 * consume.  It holds none of the matmul's arithmetic: it only draws numbers
 * and writes them in the packed storage format.  Every value depends only on
 * (seed, tensor id, element index), so any sub-range can be regenerated on its
 * own and the result does not depend on the number of threads used.
 *
 * Counter hash.  The i-th value of tensor `tid` under `seed` is the (i+1)-th
 * output of a splitmix64 generator (Steele, Lea, Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) whose state starts at
 *     key = mix(seed XOR (tid * 0xD1B54A32D192ED03))
 * where mix() is the splitmix64 output function.  Hence
 *     h(seed, tid, i) = mix(key + (i + 1) * 0x9E3779B97F4A7C15).
 *
 * Distributions (the workloads of the pages, see the header of each call):
 *   uniform u    = (h >> 40) * 2^-24                     in [0, 1)
 *   normal  z    = Box-Muller on h(.., 2i) and h(.., 2i+1) in fp64
 *   bf16(v)      = IEEE round-to-nearest-even of the fp32 value (float)v
 *
 * Tensor ids: x = 1, packed codes = 2, scales = 3, bias noise = 4, ids = 5,
 * STQ1_0 code and sign bytes = 6, STQ1_0 scales = 7.
 *
 * Ownership: every pointer is a HOST pointer owned by the caller; the
 * library allocates nothing and keeps no state.  Calls are thread-safe.
 * Return value: 0 on success, -1 on a null pointer, -2 on a negative size.
 */
#ifndef W4A16_SYNTH_H
#define W4A16_SYNTH_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  W4A16_SYNTH_TID_X = 1,
  W4A16_SYNTH_TID_CODES = 2,
  W4A16_SYNTH_TID_SCALES = 3,
  W4A16_SYNTH_TID_BIAS_NOISE = 4,
  W4A16_SYNTH_TID_IDS = 5,
  W4A16_SYNTH_TID_STQ1_BITS = 6,
  W4A16_SYNTH_TID_STQ1_SCALE = 7
};

/* Raw counter hash h(seed, tid, i) for i in [offset, offset + n). */
int w4a16_synth_hash(uint64_t seed, uint32_t tid, uint64_t offset, int64_t n,
                     uint64_t* out);

/* Activations: out[i] = bf16(N(0,1) draw number offset+i of tensor id 1).
 * Row-major x[M][K] is the call with offset = 0 and n = M*K. */
int w4a16_synth_x(uint64_t seed, uint64_t offset, int64_t n, uint16_t* out);

/* Packed codes: out[i] = high 32 bits of h(seed, 2, offset + i).  Each word
 * holds 8 codes, low nibble first; every nibble is uniform on 0..15 and the
 * nibbles are independent.  Row-major Wq[N][K/8] is offset = 0, n = N*K/8. */
int w4a16_synth_codes(uint64_t seed, uint64_t offset, int64_t n, uint32_t* out);

/* Group parameters for elements [offset, offset + n) of scales[N][K/64]:
 *   scale = bf16(0.002 + 0.018 * u)                 (u from tensor id 3)
 *   bias  = bf16((float)(-8 * scale + 1e-3 * z))    (z from tensor id 4)
 * Either output pointer may be NULL to skip it. */
int w4a16_synth_group_params(uint64_t seed, uint64_t offset, int64_t n,
                             uint16_t* scales, uint16_t* biases);

/* Expert ids: out[t] = floor(E * (h(seed, 5, t) >> 32) / 2^32), uniform on
 * 0..E-1.  Returns -2 if E <= 0. */
int w4a16_synth_ids(uint64_t seed, int64_t T, int32_t E, int32_t* out);

/* Float32 activations: out[i] = (float)(N(0,1) draw number offset+i of
 * tensor id 1) -- the draws of w4a16_synth_x before their bf16 rounding. */
int w4a16_synth_x_f32(uint64_t seed, uint64_t offset, int64_t n, float* out);

/* STQ1_0 blocks of the "Hy4-preview Metal kernels for llama.cpp" page
 * (section "Notes and gotchas"), 42 bytes each, for blocks
 * [offset, offset + n) of a row-major [N][K/256] block matrix:
 *   bytes 0..39  = little-endian bytes of h(seed, 6, 5*blk + w), w = 0..4
 *                  (32 bytes of 4-bit group codes, then 8 bytes of group
 *                  sign bits: every code uniform on 0..15, every sign bit
 *                  uniform, all independent),
 *   bytes 40..41 = fp16(0.002 + 0.018 * u), u from h(seed, 7, blk), little
 *                  endian (finite, as the page's "Test-data hygiene" asks).
 * out must hold 42 * n bytes. */
int w4a16_synth_stq1(uint64_t seed, uint64_t offset, int64_t n, uint8_t* out);

/* fp16 bits of v, IEEE round to nearest even (the encoder the blocks use). */
int w4a16_synth_fp16(float v, uint16_t* out);

/* Number of host threads the generator uses (all online cores, <= 64). */
int w4a16_synth_threads(void);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_SYNTH_H */

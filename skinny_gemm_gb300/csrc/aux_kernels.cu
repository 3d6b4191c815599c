// aux_kernels.cu -- the readable control kernel and the bit-exact debug kernels.
//
// Citations (page titles; sections in quotes):
//   [W2D2] tiny-llm book, "Week 2 Day 2: Keep W4 Packed"
//
// vanilla: one thread per output element, walking groups, packs and nibbles
// in the order of [W2D2 "Computation Flow"] with an fp32 accumulator and no
// sharing between threads ([W2D2 "Stage 1: Vanilla Matmul": an inspectable
// bring-up control).  It is a debug control, not a timed path.
//
// unpack / dequant: the debug outputs the page recommends comparing first
// ([W2D2 "Make Failures Small and Synchronous": compare an intermediate such
// as a dequantized weight group).  dequant computes fp32 fma(q, s, b) with a
// single rounding.
//
// embed: the quantized embedding row lookup of [W2D2] "Task 1: Implement
// Quantized Linear and Embedding" (gather the selected packed rows, unpack,
// q * scale + bias): the same single-rounding fp32 fma as dequant, then the
// output's round-to-nearest-even to bf16.
//
// expand_groups: scales or biases of a table quantized with a larger group
// (the book's 128 codes per scale and bias) repeated over its 64-code halves,
// so that the group-64 kernels compute q * s + b with the same s and b.
#include "common.cuh"
#include "launch.h"

namespace w4a16 {
namespace {

__device__ __forceinline__ float vanilla_dot(const uint16_t* __restrict__ xrow, const uint32_t* __restrict__ Wq,
                                             const uint16_t* __restrict__ S, const uint16_t* __restrict__ B, int K,
                                             int n) {
  const int64_t words_per_row = K / 8, groups = K / kGroup;
  float sum = 0.0f;
  for (int g = 0; g < groups; ++g) {
    const float scale = bf16_bits_to_f32(S[n * groups + g]);
    const float bias = bf16_bits_to_f32(B[n * groups + g]);
    for (int p = 0; p < kGroup / 8; ++p) {
      const uint32_t packed = Wq[n * words_per_row + g * (kGroup / 8) + p];
      for (int bit = 0; bit < 32; bit += 4) {
        const float q = (float)((packed >> bit) & 0xFu);
        const float w = __fmaf_rn(q, scale, bias);
        const float a = bf16_bits_to_f32(xrow[g * kGroup + p * 8 + bit / 4]);
        sum = __fmaf_rn(a, w, sum);
      }
    }
  }
  return sum;
}

__global__ void vanilla_mm_kernel(const uint16_t* __restrict__ x, const uint32_t* __restrict__ Wq,
                                  const uint16_t* __restrict__ S, const uint16_t* __restrict__ B,
                                  uint16_t* __restrict__ y, int row0, int N, int K) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  const int m = row0 + blockIdx.y;
  if (n >= N) return;
  y[(int64_t)m * N + n] = f32_to_bf16_bits(vanilla_dot(x + (int64_t)m * K, Wq, S, B, K, n));
}

__global__ void vanilla_mm_id_kernel(const uint16_t* __restrict__ x, const uint32_t* __restrict__ Wq,
                                     const uint16_t* __restrict__ S, const uint16_t* __restrict__ B,
                                     const int32_t* __restrict__ ids, uint16_t* __restrict__ y, int N, int K, int E,
                                     int* flags) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  const int t = blockIdx.y;
  if (n >= N) return;
  const int e = ids[t];
  if (e < 0 || e >= E) {
    y[(int64_t)t * N + n] = 0;
    if (n == 0) atomicOr(flags, W4A16_DEVICE_BAD_ID);
    return;
  }
  const int64_t words = (int64_t)N * (K / 8), params = (int64_t)N * (K / kGroup);
  y[(int64_t)t * N + n] =
      f32_to_bf16_bits(vanilla_dot(x + (int64_t)t * K, Wq + e * words, S + e * params, B + e * params, K, n));
}

__global__ void unpack_kernel(const uint32_t* __restrict__ Wq, uint8_t* __restrict__ q, int64_t nwords) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nwords) return;
  const uint32_t w = Wq[i];
  uint2 out;
  out.x = (w & 0xFu) | ((w >> 4) & 0xFu) << 8 | ((w >> 8) & 0xFu) << 16 | ((w >> 12) & 0xFu) << 24;
  out.y = ((w >> 16) & 0xFu) | ((w >> 20) & 0xFu) << 8 | ((w >> 24) & 0xFu) << 16 | ((w >> 28) & 0xFu) << 24;
  reinterpret_cast<uint2*>(q)[i] = out;
}

__global__ void dequant_kernel(const uint32_t* __restrict__ Wq, const uint16_t* __restrict__ S,
                               const uint16_t* __restrict__ B, float* __restrict__ w, int64_t nwords, int K) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nwords) return;
  const int64_t words_per_row = K / 8;
  const int64_t n = i / words_per_row, k0 = (i % words_per_row) * 8;
  const int64_t gi = n * (K / kGroup) + k0 / kGroup;
  const float s = bf16_bits_to_f32(S[gi]), b = bf16_bits_to_f32(B[gi]);
  const uint32_t word = Wq[i];
  float4 lo, hi;
  lo.x = __fmaf_rn((float)((word >> 0) & 0xFu), s, b);
  lo.y = __fmaf_rn((float)((word >> 4) & 0xFu), s, b);
  lo.z = __fmaf_rn((float)((word >> 8) & 0xFu), s, b);
  lo.w = __fmaf_rn((float)((word >> 12) & 0xFu), s, b);
  hi.x = __fmaf_rn((float)((word >> 16) & 0xFu), s, b);
  hi.y = __fmaf_rn((float)((word >> 20) & 0xFu), s, b);
  hi.z = __fmaf_rn((float)((word >> 24) & 0xFu), s, b);
  hi.w = __fmaf_rn((float)((word >> 28) & 0xFu), s, b);
  reinterpret_cast<float4*>(w)[2 * i] = lo;
  reinterpret_cast<float4*>(w)[2 * i + 1] = hi;
}

// One thread per packed word (eight codes) of token t's row; grid.y = token.
// 16 bytes of bf16 out per thread.  An id outside 0..N-1 gives a zero row
// and raises the device flag.
__global__ void embed_kernel(const uint32_t* __restrict__ Wq, const uint16_t* __restrict__ S,
                             const uint16_t* __restrict__ B, const int32_t* __restrict__ ids, uint16_t* __restrict__ out,
                             int N, int K, int* flags) {
  const int t = blockIdx.y;
  const int words = K / 8;
  const int wi = blockIdx.x * blockDim.x + threadIdx.x;
  if (wi >= words) return;
  const int n = ids[t];
  uint4 v = make_uint4(0, 0, 0, 0);
  if (n < 0 || n >= N) {
    if (wi == 0) atomicOr(flags, W4A16_DEVICE_BAD_ID);
  } else {
    const int64_t gi = (int64_t)n * (K / kGroup) + (8 * wi) / kGroup;
    const float s = bf16_bits_to_f32(S[gi]), b = bf16_bits_to_f32(B[gi]);
    const uint32_t word = Wq[(int64_t)n * words + wi];
    uint32_t h[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] = f32_to_bf16_bits(__fmaf_rn((float)((word >> (4 * i)) & 0xFu), s, b));
    v = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
  }
  reinterpret_cast<uint4*>(out + (int64_t)t * K)[wi] = v;
}

__global__ void expand_groups_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst, int64_t n64,
                                     int rep) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n64) dst[i] = src[i / rep];
}

}  // namespace

void plan_vanilla(int N, int K, w4a16_plan* p) {
  (void)K;
  p->kernel = W4A16_KERNEL_VANILLA;
  p->ksplit = 1;
  p->slice_k = K;
  p->rows_per_tile = 128;
  p->threads = 128;
  p->grid_x = (N + 127) / 128;
  p->units = p->grid_x;
  p->smem_bytes = 0;
  p->workspace_bytes = 0;
}

cudaError_t launch_vanilla(const LaunchArgs& a, const w4a16_plan& p) {
  dim3 grid(p.grid_x, a.M);
  vanilla_mm_kernel<<<grid, p.threads, 0, a.stream>>>(a.x, a.Wq, a.S, a.B, a.y, a.row0, a.N, a.K);
  return cudaGetLastError();
}

cudaError_t launch_vanilla_id(const LaunchArgs& a, const w4a16_plan& p) {
  dim3 grid(p.grid_x, a.T);
  vanilla_mm_id_kernel<<<grid, p.threads, 0, a.stream>>>(a.x, a.Wq, a.S, a.B, a.ids, a.y, a.N, a.K, a.E, a.flags);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint32_t* Wq, uint8_t* q, int N, int K, cudaStream_t s) {
  const int64_t nwords = (int64_t)N * (K / 8);
  const int threads = 256;
  const int64_t blocks = (nwords + threads - 1) / threads;
  unpack_kernel<<<(unsigned)blocks, threads, 0, s>>>(Wq, q, nwords);
  return cudaGetLastError();
}

cudaError_t launch_embed(const uint32_t* Wq, const uint16_t* S, const uint16_t* B, const int32_t* ids,
                         uint16_t* out, int T, int N, int K, int* flags, cudaStream_t s) {
  const int threads = 128;
  const dim3 grid((unsigned)((K / 8 + threads - 1) / threads), (unsigned)T);
  embed_kernel<<<grid, threads, 0, s>>>(Wq, S, B, ids, out, N, K, flags);
  return cudaGetLastError();
}

cudaError_t launch_expand_groups(const uint16_t* src, uint16_t* dst, int N, int K, int group, cudaStream_t s) {
  const int64_t n64 = (int64_t)N * (K / kGroup);
  const int threads = 256;
  const int64_t blocks = (n64 + threads - 1) / threads;
  expand_groups_kernel<<<(unsigned)blocks, threads, 0, s>>>(src, dst, n64, group / kGroup);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const uint32_t* Wq, const uint16_t* S, const uint16_t* B, float* w, int N, int K,
                           cudaStream_t s) {
  const int64_t nwords = (int64_t)N * (K / 8);
  const int threads = 256;
  const int64_t blocks = (nwords + threads - 1) / threads;
  dequant_kernel<<<(unsigned)blocks, threads, 0, s>>>(Wq, S, B, w, nwords, K);
  return cudaGetLastError();
}

}  // namespace w4a16

// simt.cu -- CUDA-core W4A16 skinny GEMM: fp32 FMA accumulation and a
// warp-shuffle split-K reduction, specialised for M = 1..8.
//
// Citations (page titles; sections in quotes):
//   [W2D2] tiny-llm book, "Week 2 Day 2: Keep W4 Packed"
//   [G4MK] "Gemma 4 E4B & E2B -- single-launch Metal megakernels + lossless
//          speculative decoding" (RESMP-DEV model card)
//   [HY4]  "Hy4-preview Metal kernels for llama.cpp"
//
// Schedule.  A warp owns four output rows ([G4MK "Implementation notes":
// four output rows per SIMD group for memory-level parallelism) and
// reduces K cooperatively ([W2D2 "Stage 2: SIMD Matvec": the SIMD group
// reduces the input dimension, simd_sum combines lane partials).  Each lane
// streams one 16-byte packed chunk (32 codes = half a 64-group) per row per
// step, so a warp step reads 512 contiguous bytes of each row.  `ksplit`
// warps share a row tile and take interleaved K steps; their partials meet
// in shared memory and are added in warp order.
//
// Arithmetic per lane and step, for every row r and activation row m
// ([W2D2 "Stage 2: SIMD Matvec", the affine identity
//  sum a(sq+b) = s*sum(a q) + b*sum(a)):
//   P[r][m] = sum over the lane's 32 codes of x*q      (fixed order)
//   X[m]    = sum over the same 32 activations          (fixed order)
//   acc[r][m] = fma(s, P, acc);  acc[r][m] = fma(b, X, acc)
// then a butterfly over lanes (xor 16, 8, 4, 2, 1) and the cross-warp sum,
// then round to bf16 ([W2D2 "Computation Flow": C = bfloat16(sum)).
//
// Batch invariance: every value above depends only on its own row m and on
// K through ksplit; the same fp32 operations run in the same order for
// every M (explicit __fmaf_rn / __fadd_rn, compiled with -fmad=false), so
// row m of an M-row launch equals the M = 1 launch bit for bit.
#include "common.cuh"
#include "launch.h"
#include "route.cuh"

namespace w4a16 {
namespace {

constexpr int kRowsPerWarp = 4;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStepK = 32 * 32;        // codes per warp step (32 lanes x 32 codes)

template <int M>
__device__ __forceinline__ void simt_tile(const uint16_t* __restrict__ x, const uint32_t* __restrict__ Wq,
                                          const uint16_t* __restrict__ S, const uint16_t* __restrict__ B,
                                          uint16_t* __restrict__ y, int N, int K, int ksplit, int tile,
                                          const int* s_row, float* s_red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows_per_cta = kRowsPerWarp * (kWarps / ksplit);
  const int rg = warp / ksplit, ks = warp % ksplit;
  const int rbase = tile * rows_per_cta + rg * kRowsPerWarp;
  const int64_t words_per_row = K / 8, groups = K / kGroup;

  int xr[M];
#pragma unroll
  for (int m = 0; m < M; ++m) xr[m] = s_row[m];

  float acc[kRowsPerWarp][M];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) acc[r][m] = 0.0f;

  for (int s = ks; s * kStepK < K; s += ksplit) {
    const int k0 = s * kStepK + lane * 32;
    if (k0 < K) {
      uint4 wv[kRowsPerWarp];
      float sc[kRowsPerWarp], bi[kRowsPerWarp];
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) {
        const int row = rbase + r;
        if (row < N) {
          wv[r] = ld_stream_v4(Wq + row * words_per_row + k0 / 8);
          sc[r] = bf16_bits_to_f32(ld_nc_u16(S + row * groups + k0 / kGroup));
          bi[r] = bf16_bits_to_f32(ld_nc_u16(B + row * groups + k0 / kGroup));
        } else {
          wv[r] = make_uint4(0, 0, 0, 0);
          sc[r] = 0.0f;
          bi[r] = 0.0f;
        }
      }
      float P[kRowsPerWarp][M], X[M];
#pragma unroll
      for (int m = 0; m < M; ++m) {
        X[m] = 0.0f;
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) P[r][m] = 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float xf[M][8];
#pragma unroll
        for (int m = 0; m < M; ++m) {
          widen8(ld_nc_v4(x + (int64_t)xr[m] * K + k0 + 8 * i), xf[m]);
#pragma unroll
          for (int j = 0; j < 8; ++j) X[m] = __fadd_rn(X[m], xf[m][j]);
        }
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
          float q[8];
          unpack8_f32(word_of(wv[r], i), q);
#pragma unroll
          for (int m = 0; m < M; ++m)
#pragma unroll
            for (int j = 0; j < 8; ++j) P[r][m] = __fmaf_rn(xf[m][j], q[j], P[r][m]);
        }
      }
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) {
          acc[r][m] = __fmaf_rn(sc[r], P[r][m], acc[r][m]);
          acc[r][m] = __fmaf_rn(bi[r], X[m], acc[r][m]);
        }
    }
  }

  // Butterfly over the 32 lanes; IEEE addition is commutative, so every lane
  // ends with the same sum.
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float v = acc[r][m];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
      acc[r][m] = v;
    }
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
      for (int m = 0; m < M; ++m) s_red[((rg * kRowsPerWarp + r) * M + m) * ksplit + ks] = acc[r][m];
  }
  __syncthreads();
  for (int t = threadIdx.x; t < rows_per_cta * M; t += blockDim.x) {
    const int rr = t / M, m = t % M;
    const float* part = s_red + (rr * M + m) * ksplit;
    float sum = part[0];
    for (int j = 1; j < ksplit; ++j) sum = __fadd_rn(sum, part[j]);
    const int row = tile * rows_per_cta + rr;
    if (row < N) y[(int64_t)s_row[m] * N + row] = f32_to_bf16_bits(sum);
  }
  __syncthreads();
}

template <int M>
__global__ void __launch_bounds__(kThreads) simt_mm_kernel(const uint16_t* __restrict__ x,
                                                           const uint32_t* __restrict__ Wq,
                                                           const uint16_t* __restrict__ S,
                                                           const uint16_t* __restrict__ B,
                                                           uint16_t* __restrict__ y, int row0, int N, int K,
                                                           int ksplit) {
  __shared__ int s_row[kMaxChunk];
  __shared__ float s_red[kRowsPerWarp * kWarps * kMaxChunk];
  if (threadIdx.x < M) s_row[threadIdx.x] = row0 + threadIdx.x;
  __syncthreads();
  simt_tile<M>(x, Wq, S, B, y, N, K, ksplit, blockIdx.x, s_row, s_red);
}

__global__ void __launch_bounds__(kThreads) simt_mm_id_kernel(const uint16_t* __restrict__ x,
                                                              const uint32_t* __restrict__ Wq,
                                                              const uint16_t* __restrict__ S,
                                                              const uint16_t* __restrict__ B,
                                                              const int32_t* __restrict__ ids,
                                                              uint16_t* __restrict__ y, int T, int N, int K,
                                                              int E, int ksplit, int* flags) {
  __shared__ int s_tok[kMaxChunk];
  __shared__ int s_state[2];
  __shared__ float s_red[kRowsPerWarp * kWarps * kMaxChunk];
  const int e = blockIdx.y;
  const int64_t words = (int64_t)N * (K / 8), params = (int64_t)N * (K / kGroup);
  const uint32_t* We = Wq + e * words;
  const uint16_t* Se = S + e * params;
  const uint16_t* Be = B + e * params;
  if (threadIdx.x == 0) s_state[0] = 0;
  __syncthreads();
  for (;;) {
    const int cnt = gather_tokens(ids, T, E, e, s_tok, s_state);
    if (cnt == 0) break;
    switch (cnt) {
      case 1: simt_tile<1>(x, We, Se, Be, y, N, K, ksplit, blockIdx.x, s_tok, s_red); break;
      case 2: simt_tile<2>(x, We, Se, Be, y, N, K, ksplit, blockIdx.x, s_tok, s_red); break;
      case 3: simt_tile<3>(x, We, Se, Be, y, N, K, ksplit, blockIdx.x, s_tok, s_red); break;
      case 4: simt_tile<4>(x, We, Se, Be, y, N, K, ksplit, blockIdx.x, s_tok, s_red); break;
      case 5: simt_tile<5>(x, We, Se, Be, y, N, K, ksplit, blockIdx.x, s_tok, s_red); break;
      case 6: simt_tile<6>(x, We, Se, Be, y, N, K, ksplit, blockIdx.x, s_tok, s_red); break;
      case 7: simt_tile<7>(x, We, Se, Be, y, N, K, ksplit, blockIdx.x, s_tok, s_red); break;
      default: simt_tile<8>(x, We, Se, Be, y, N, K, ksplit, blockIdx.x, s_tok, s_red); break;
    }
  }
  if (e == 0) {
    // Tokens whose id is out of range: zero rows of this tile, raise the flag.
    const int rows_per_cta = kRowsPerWarp * (kWarps / ksplit);
    if (threadIdx.x == 0) s_state[0] = 0;
    __syncthreads();
    for (;;) {
      const int cnt = gather_tokens(ids, T, E, -1, s_tok, s_state);
      if (cnt == 0) break;
      if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(flags, W4A16_DEVICE_BAD_ID);
      for (int t = threadIdx.x; t < cnt * rows_per_cta; t += blockDim.x) {
        const int row = blockIdx.x * rows_per_cta + t % rows_per_cta;
        if (row < N) y[(int64_t)s_tok[t / rows_per_cta] * N + row] = 0;
      }
      __syncthreads();
    }
  }
}

template <int M>
cudaError_t launch_m(const LaunchArgs& a, const w4a16_plan& p) {
  simt_mm_kernel<M><<<p.grid_x, p.threads, 0, a.stream>>>(a.x, a.Wq, a.S, a.B, a.y, a.row0, a.N, a.K, p.ksplit);
  return cudaGetLastError();
}

}  // namespace

// The reduction order (ksplit) depends on K alone, so a row's result does not
// depend on N either: splitting the output rows over several launches (or
// GPUs) reproduces the unsplit call bit for bit.
void plan_simt(int N, int K, w4a16_plan* p) {
  const int steps = (K + kStepK - 1) / kStepK;
  int ks = 1;
  while (ks < kWarps && ks * 2 <= steps) ks *= 2;
  const int rows_per_cta = kRowsPerWarp * (kWarps / ks);
  p->kernel = W4A16_KERNEL_SIMT;
  p->ksplit = ks;  // warps interleaving K steps of kStepK codes
  p->slice_k = kStepK;
  p->rows_per_tile = rows_per_cta;
  p->threads = kThreads;
  p->grid_x = (int)((N + rows_per_cta - 1) / rows_per_cta);
  p->units = p->grid_x;
  p->smem_bytes = 0;
  p->workspace_bytes = 0;
}

cudaError_t launch_simt(const LaunchArgs& a, const w4a16_plan& p) {
  switch (a.M) {
    case 1: return launch_m<1>(a, p);
    case 2: return launch_m<2>(a, p);
    case 3: return launch_m<3>(a, p);
    case 4: return launch_m<4>(a, p);
    case 5: return launch_m<5>(a, p);
    case 6: return launch_m<6>(a, p);
    case 7: return launch_m<7>(a, p);
    case 8: return launch_m<8>(a, p);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_simt_id(const LaunchArgs& a, const w4a16_plan& p) {
  dim3 grid(p.grid_x, a.E);
  simt_mm_id_kernel<<<grid, p.threads, 0, a.stream>>>(a.x, a.Wq, a.S, a.B, a.ids, a.y, a.T, a.N, a.K, a.E,
                                                      p.ksplit, a.flags);
  return cudaGetLastError();
}

}  // namespace w4a16

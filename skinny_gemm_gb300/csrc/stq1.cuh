// stq1.cuh -- internal interface between the C-ABI (api.cu) and the STQ1_0
// kernels (stq1.cu).  Host-side only.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace w4a16 {

struct Stq1Plan {
  int nb;      // 256-weight blocks per row
  int tiles;   // 16-row tiles
  int ks;      // K slices per tile (1, 2, 4 or 8)
  int bps;     // blocks per slice
  int rt;      // tiles per round of one CTA (8 / ks)
  int rounds;  // ceil(tiles / rt)
  int xcap;    // activation rows staged per pass
};

bool stq1_shape_ok(int N, int K);
void stq1_make_plan(int N, int K, Stq1Plan* p);
size_t stq1_packed_size(int N, int K);

cudaError_t launch_stq1_pack(const uint8_t* src, uint8_t* dst, int N, int K, cudaStream_t s);
// One pass: rows row0 .. row0 + M - 1 (M <= plan.xcap).
cudaError_t launch_stq1_mm(const float* x, const uint8_t* w, float* y, int M, int row0, int N, int K,
                           cudaStream_t s);
cudaError_t launch_stq1_mm_id(const float* x, const uint8_t* w, const int32_t* ids, float* y, int T, int N,
                              int K, int E, int* flags, cudaStream_t s);
cudaError_t launch_stq1_get_rows(const uint8_t* w, const int32_t* ids, float* out, int T, int N, int K,
                                 int* flags, cudaStream_t s);

}  // namespace w4a16

// stq1.cuh -- internal interface between the C-ABI (api.cu) and the STQ1_0
// kernels (stq1.cu).  Host-side only.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace w4a16 {

struct Stq1Plan {
  int nb;       // 256-weight blocks per row
  int tiles;    // 16-row tiles (records per block column)
  int rgroups;  // 256-row groups (one cluster each)
  int ks;       // K slices: CTAs of a cluster (1 .. 8)
  int bps;      // blocks per slice (the last may have fewer)
  int xcap;     // activation rows per pass
};

bool stq1_shape_ok(int N, int K);
void stq1_make_plan(int N, int K, Stq1Plan* p);
size_t stq1_packed_size(int N, int K);

cudaError_t launch_stq1_pack(const uint8_t* src, uint8_t* dst, int N, int K, cudaStream_t s);
// One pass: rows row0 .. row0 + M - 1 (M <= plan.xcap).
// pdl: W4A16_PDL (0 plain launches, 1 overlapped, 2 also the first records
// requested before the wait for earlier kernels).
cudaError_t launch_stq1_mm(const float* x, const uint8_t* w, float* y, int M, int row0, int N, int K, int* flags,
                           int pdl, cudaStream_t s);
cudaError_t launch_stq1_mm_id(const float* x, const uint8_t* w, const int32_t* ids, float* y, int T, int N,
                              int K, int E, int* flags, int pdl, cudaStream_t s);
cudaError_t launch_stq1_get_rows(const uint8_t* w, const int32_t* ids, float* out, int T, int N, int K,
                                 int* flags, cudaStream_t s);

}  // namespace w4a16

// launch.h -- internal interface between the C-ABI (api.cu) and the kernel
// translation units.  Host-side only; no torch types anywhere.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "w4a16.h"

namespace w4a16 {

// One launch computes at most this many activation rows.
constexpr int kMaxChunk = 8;

// Arguments of one launch.  Plain mm: rows x[row0 .. row0+M) -> y rows of the
// same index.  Routed mm_id: ids != nullptr, T tokens, E experts; each CTA
// column blockIdx.y is one expert and gathers its own tokens.
struct LaunchArgs {
  const uint16_t* x;
  const uint32_t* Wq;
  const uint16_t* S;
  const uint16_t* B;
  uint16_t* y;
  int M;          // rows (1..8 for the CUDA-core and control kernels; any for the tensor-core
                  // family, which takes them eight at a time); unused for mm_id
  int row0;       // first activation row of the chunk
  int N, K;
  const int32_t* ids;  // mm_id only
  int T, E;            // mm_id only
  int* flags;          // device flag word (mm_id bad ids)
  int pdl;             // 0: plain launch; 1: programmatic dependent launch; 2: and weights fetched before the wait
  int tc_path;         // tensor-core launch shape: 0 the dispatcher's choice, 1 persistent, 2 tile
  cudaStream_t stream;
  void* ws = nullptr;  // the caller's workspace (w4a16_mm_ws, w4a16_mm_argmax), or none
  size_t ws_bytes = 0;
  int fault_wait = 0;  // debug (W4A16_FAULT=wait): the persistent kernel's first stage never completes
};

// Per-family planning (depends on N and K only) and launching.
void plan_simt(int N, int K, w4a16_plan* p);
cudaError_t launch_simt(const LaunchArgs& a, const w4a16_plan& p);
cudaError_t launch_simt_id(const LaunchArgs& a, const w4a16_plan& p);

// tc_path: 0 the dispatcher's choice, 1 the persistent grid, 2 the tile kernel.
void plan_tc(int N, int K, int tc_path, w4a16_plan* p);
bool tc_supported(int N, int K);
bool tc_tile_fits(int N, int K, int M);
cudaError_t launch_tc(const LaunchArgs& a, const w4a16_plan& p);
cudaError_t launch_tc_id(const LaunchArgs& a, const w4a16_plan& p);
// w4a16_mm_argmax: the persistent kernel in argmax mode (rows a.row0 .. a.row0 + a.M).
cudaError_t launch_tc_argmax(const LaunchArgs& a, int32_t* idx, uint16_t* val);
// Grouped tensor-core launch (w4a16_mm_group): items sharing K and M.
struct GroupItem {
  const uint16_t* x;
  const uint32_t* Wq;
  const uint16_t* S;
  const uint16_t* B;
  uint16_t* y;
  int N;
};
bool tc_group_supported(const int* N, int count, int K);
// M rows in one launch, eight at a time over resident weights.
cudaError_t launch_tc_group(const GroupItem* items, int count, int M, int row0, int K, int pdl, int* flags,
                            cudaStream_t stream);
// A 2-D TMA tensor map of a row-major tensor (`inner` elements per row,
// `outer` rows, rows `row_bytes` apart) with boxes of box_inner x box_outer.
cudaError_t encode_map_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, int64_t inner,
                          int64_t outer, int64_t row_bytes, int box_inner, int box_outer, CUtensorMapSwizzle swizzle);
// Activation rows from which w4a16_mm runs the tcgen05 prefill kernel (below,
// the skinny tile kernel taking eight rows at a time is faster).
constexpr int kPrefillMinM = 33;
// The tcgen05 prefill kernel (prefill.cu): rows a.row0 .. a.row0 + a.M, the
// canonical slices of slice_k codes.
cudaError_t launch_prefill(const LaunchArgs& a, int slice_k);
// w4a16_mm_g with group 128: the persistent kernel reading [N][K/128] tables.
cudaError_t launch_tc_g128(const LaunchArgs& a);
// Bytes of the persistent kernel's workspace (counters, split-K partials, argmax keys).
size_t tc_workspace_bytes();
// Tensor-core w4a16_mm with its split-K scratch in a fixed device array (no allocation).
cudaError_t launch_tc_noalloc(const LaunchArgs& a);
size_t tc_noalloc_scratch_bytes();
bool tc_noalloc_fits(int N, int K);

void plan_vanilla(int N, int K, w4a16_plan* p);
cudaError_t launch_vanilla(const LaunchArgs& a, const w4a16_plan& p);
cudaError_t launch_vanilla_id(const LaunchArgs& a, const w4a16_plan& p);

cudaError_t launch_unpack(const uint32_t* Wq, uint8_t* q, int N, int K, cudaStream_t s);
cudaError_t launch_dequant(const uint32_t* Wq, const uint16_t* S, const uint16_t* B, float* w, int N, int K,
                           cudaStream_t s);
cudaError_t launch_expand_groups(const uint16_t* src, uint16_t* dst, int N, int K, int group, cudaStream_t s);
cudaError_t launch_embed(const uint32_t* Wq, const uint16_t* S, const uint16_t* B, const int32_t* ids,
                         uint16_t* out, int T, int N, int K, int* flags, cudaStream_t s);

}  // namespace w4a16

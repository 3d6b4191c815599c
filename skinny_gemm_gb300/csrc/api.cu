// api.cu -- the C ABI of libw4a16.so (declared and documented in include/w4a16.h).
//
// Host-side validation happens before any launch and a rejected call writes
// nothing (fail closed, after tiny-llm "Week 2 Day 2: Keep W4 Packed",
// section "Task 2": validate inputs, reject unsupported evaluation
// explicitly).  The kernel family and its reduction order are chosen from
// (N, K) only; M only decides how many chunks of at most eight rows run.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "common.cuh"
#include "launch.h"
#include "stq1.cuh"
#include "stq1.h"

namespace w4a16 {
namespace {

__device__ int g_device_flags;

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(W4A16_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

// ---- debug switches read once from the environment -----------------------------

enum Fault { kFaultNone = 0, kFaultValidate = 1, kFaultLaunch = 2, kFaultWait = 3 };

struct EnvConfig {
  int fault = kFaultNone;
  int force_kernel = W4A16_KERNEL_AUTO;
  int pdl = 2;  // W4A16_PDL: 0 plain launches, 1 overlap launches only, 2 also fetch weights early
};

std::mutex g_env_mu;
bool g_env_loaded = false;
EnvConfig g_env;

void load_env_locked() {
  EnvConfig c;
  if (const char* f = std::getenv("W4A16_FAULT")) {
    if (!std::strcmp(f, "validate")) c.fault = kFaultValidate;
    else if (!std::strcmp(f, "launch")) c.fault = kFaultLaunch;
    else if (!std::strcmp(f, "wait")) c.fault = kFaultWait;
  }
  if (const char* v = std::getenv("W4A16_PDL")) {
    if (v[0] >= '0' && v[0] <= '2' && v[1] == 0) c.pdl = v[0] - '0';
  }
  if (const char* k = std::getenv("W4A16_FORCE_KERNEL")) {
    if (!std::strcmp(k, "simt")) c.force_kernel = W4A16_KERNEL_SIMT;
    else if (!std::strcmp(k, "tc")) c.force_kernel = W4A16_KERNEL_TC;
    else if (!std::strcmp(k, "vanilla")) c.force_kernel = W4A16_KERNEL_VANILLA;
  }
  g_env = c;
  g_env_loaded = true;
}

EnvConfig env() {
  std::lock_guard<std::mutex> lk(g_env_mu);
  if (!g_env_loaded) load_env_locked();
  return g_env;
}

// ---- device flag word, one per device ------------------------------------------

constexpr int kMaxDevices = 64;
std::mutex g_flag_mu;
int* g_flag_ptr[kMaxDevices] = {};

int flag_pointer(int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(W4A16_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_flag_mu);
  if (!g_flag_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_flags);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(device flags)");
    g_flag_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_flag_ptr[dev];
  return W4A16_OK;
}

// ---- validation ------------------------------------------------------------------

constexpr int kMaxDim = 1 << 30;

bool misaligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; }

int check_nk(int N, int K) {
  if (N <= 0 || N > kMaxDim) return fail(W4A16_ERR_SHAPE, "N = %d must be in 1..2^30", N);
  if (K <= 0 || K > kMaxDim || K % kGroup) return fail(W4A16_ERR_SHAPE, "K = %d must be a positive multiple of 64", K);
  return W4A16_OK;
}

int resolve_kernel(int requested, int N, int K, w4a16_plan* plan) {
  int k = requested;
  if (k == W4A16_KERNEL_AUTO) k = env().force_kernel;
  // Default: the tensor-core family wherever it applies (K % 512 == 0, and
  // K % 512 != 0 padded to whole 512-code stages up to the K whose per-unit
  // parameter rows fit in shared memory), the CUDA-core family otherwise.
  // The choice depends on (N, K) only.
  if (k == W4A16_KERNEL_AUTO) k = tc_supported(N, K) ? W4A16_KERNEL_TC : W4A16_KERNEL_SIMT;
  switch (k) {
    case W4A16_KERNEL_SIMT: plan_simt(N, K, plan); return W4A16_OK;
    case W4A16_KERNEL_VANILLA: plan_vanilla(N, K, plan); return W4A16_OK;
    case W4A16_KERNEL_TC:
    case W4A16_KERNEL_TC_STREAM:
    case W4A16_KERNEL_TC_TILE:
    case W4A16_KERNEL_TC_PREFILL: {
      if (!tc_supported(N, K))
        return fail(W4A16_ERR_KERNEL, "K = %d is past the tensor-core kernels' K %% 512 != 0 range", K);
      if (K % 512 && k == W4A16_KERNEL_TC_PREFILL)
        return fail(W4A16_ERR_KERNEL, "the prefill kernel needs K %% 512 == 0 (K = %d)", K);
      const int path = k == W4A16_KERNEL_TC_STREAM ? 1 : k == W4A16_KERNEL_TC_TILE ? 2 : 0;
      if (path == 2 && !tc_tile_fits(N, K, 1))
        return fail(W4A16_ERR_KERNEL, "the tile kernel cannot hold K = %d in shared memory", K);
      plan_tc(N, K, path, plan);
      if (k == W4A16_KERNEL_TC_PREFILL) plan->kernel = W4A16_KERNEL_TC_PREFILL;
      return W4A16_OK;
    }
    default: return fail(W4A16_ERR_KERNEL, "unknown kernel selector %d", requested);
  }
}

int validate_mm(const void* x, const void* Wq, const void* S, const void* B, const void* y, int M, int N, int K) {
  if (M < 0 || M > kMaxDim) return fail(W4A16_ERR_SHAPE, "M = %d must be in 0..2^30", M);
  if (int rc = check_nk(N, K)) return rc;
  if (M == 0) return W4A16_OK;
  if (!x || !Wq || !S || !B || !y) return fail(W4A16_ERR_NULL, "null tensor pointer");
  if (misaligned(x, 16) || misaligned(Wq, 16)) return fail(W4A16_ERR_ALIGN, "x and Wq must be 16-byte aligned");
  if (misaligned(S, 8) || misaligned(B, 8)) return fail(W4A16_ERR_ALIGN, "scales and biases must be 8-byte aligned");
  if (misaligned(y, 2)) return fail(W4A16_ERR_ALIGN, "y must be 2-byte aligned");
  return W4A16_OK;
}

// A caller's workspace: NULL (none), or at least tc_workspace_bytes() bytes,
// 256-byte aligned.
int check_workspace(const void* ws, size_t bytes) {
  if (!ws) return W4A16_OK;
  if (misaligned(ws, 256)) return fail(W4A16_ERR_ALIGN, "the workspace must be 256-byte aligned");
  if (bytes < tc_workspace_bytes())
    return fail(W4A16_ERR_SHAPE, "a workspace of %zu bytes is too small (w4a16_workspace_bytes: %zu)", bytes,
                tc_workspace_bytes());
  return W4A16_OK;
}

int run_mm(const w4a16_bf16* x, const uint32_t* Wq, const w4a16_bf16* S, const w4a16_bf16* B, w4a16_bf16* y,
           int M, int N, int K, int kernel, void* stream, void* ws = nullptr, size_t ws_bytes = 0) {
  if (env().fault == kFaultValidate) return fail(W4A16_ERR_SHAPE, "injected validation fault (W4A16_FAULT)");
  if (int rc = validate_mm(x, Wq, S, B, y, M, N, K)) return rc;
  if (int rc = check_workspace(ws, ws_bytes)) return rc;
  w4a16_plan plan;
  if (int rc = resolve_kernel(kernel, N, K, &plan)) return rc;
  if (M == 0) return W4A16_OK;
  if (env().fault == kFaultLaunch) return fail(W4A16_ERR_CUDA, "injected launch fault (W4A16_FAULT)");
  LaunchArgs a{};
  a.x = x; a.Wq = Wq; a.S = S; a.B = B; a.y = y;
  a.N = N; a.K = K;
  a.stream = static_cast<cudaStream_t>(stream);
  a.pdl = env().pdl;
  a.tc_path = plan.kernel == W4A16_KERNEL_TC_STREAM ? 1 : plan.kernel == W4A16_KERNEL_TC_TILE ? 2
             : plan.kernel == W4A16_KERNEL_TC_PREFILL ? 3 : 0;
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  a.fault_wait = env().fault == kFaultWait;
  if (int rc = flag_pointer(&a.flags)) return rc;
  const bool tc = plan.kernel == W4A16_KERNEL_TC || plan.kernel == W4A16_KERNEL_TC_STREAM ||
                  plan.kernel == W4A16_KERNEL_TC_TILE || plan.kernel == W4A16_KERNEL_TC_PREFILL;
  if (a.tc_path == 2 && !tc_tile_fits(N, K, M < kMaxChunk ? M : kMaxChunk))
    return fail(W4A16_ERR_KERNEL, "the tile kernel cannot hold K = %d for %d rows in shared memory", K,
                M < kMaxChunk ? M : kMaxChunk);
  // The tensor-core family takes all M rows at once (the tile kernel streams
  // them over resident weights, the persistent kernel launches per chunk);
  // the CUDA-core and control kernels take chunks of at most eight rows.
  for (int row0 = 0; row0 < M; row0 += tc ? M : kMaxChunk) {
    a.row0 = row0;
    a.M = tc ? M : (M - row0 < kMaxChunk) ? M - row0 : kMaxChunk;
    cudaError_t e = cudaSuccess;
    switch (plan.kernel) {
      case W4A16_KERNEL_SIMT: e = launch_simt(a, plan); break;
      case W4A16_KERNEL_TC:
      case W4A16_KERNEL_TC_STREAM:
      case W4A16_KERNEL_TC_TILE:
      case W4A16_KERNEL_TC_PREFILL: e = launch_tc(a, plan); break;
      case W4A16_KERNEL_VANILLA: e = launch_vanilla(a, plan); break;
      default: return fail(W4A16_ERR_KERNEL, "kernel %d cannot run", plan.kernel);
    }
    if (e != cudaSuccess) return cuda_fail(e, "w4a16_mm launch");
  }
  return W4A16_OK;
}

}  // namespace
}  // namespace w4a16

using namespace w4a16;

extern "C" {

int w4a16_mm(const w4a16_bf16* x, const uint32_t* Wq, const w4a16_bf16* scales, const w4a16_bf16* biases,
             w4a16_bf16* y, int M, int N, int K, void* stream) {
  return run_mm(x, Wq, scales, biases, y, M, N, K, W4A16_KERNEL_AUTO, stream);
}

int w4a16_mm_ws(const w4a16_bf16* x, const uint32_t* Wq, const w4a16_bf16* scales, const w4a16_bf16* biases,
                w4a16_bf16* y, int M, int N, int K, void* workspace, size_t workspace_bytes, void* stream) {
  return run_mm(x, Wq, scales, biases, y, M, N, K, W4A16_KERNEL_AUTO, stream, workspace, workspace_bytes);
}

int w4a16_mm_g(const w4a16_bf16* x, const uint32_t* Wq, const w4a16_bf16* scales, const w4a16_bf16* biases,
               w4a16_bf16* y, int M, int N, int K, int group, void* workspace, size_t workspace_bytes, void* stream) {
  if (group == kGroup)
    return run_mm(x, Wq, scales, biases, y, M, N, K, W4A16_KERNEL_AUTO, stream, workspace, workspace_bytes);
  if (env().fault == kFaultValidate) return fail(W4A16_ERR_SHAPE, "injected validation fault (W4A16_FAULT)");
  if (group != 128) return fail(W4A16_ERR_SHAPE, "group = %d must be 64 or 128", group);
  if (int rc = validate_mm(x, Wq, scales, biases, y, M, N, K)) return rc;
  if (K % 512 || K > 8192)
    return fail(W4A16_ERR_SHAPE,
                "group 128 runs natively for K %% 512 == 0 up to 8192 (K = %d); expand the tables to group 64 "
                "with w4a16_expand_groups for other K", K);
  if (misaligned(scales, 16) || misaligned(biases, 16))
    return fail(W4A16_ERR_ALIGN, "group-128 scales and biases must be 16-byte aligned");
  if (int rc = check_workspace(workspace, workspace_bytes)) return rc;
  if (M == 0) return W4A16_OK;
  if (env().fault == kFaultLaunch) return fail(W4A16_ERR_CUDA, "injected launch fault (W4A16_FAULT)");
  LaunchArgs a{};
  a.x = x; a.Wq = Wq; a.S = scales; a.B = biases; a.y = y;
  a.N = N; a.K = K; a.M = M; a.row0 = 0;
  a.stream = static_cast<cudaStream_t>(stream);
  a.pdl = env().pdl;
  a.tc_path = 1;
  a.ws = workspace;
  a.ws_bytes = workspace_bytes;
  if (int rc = flag_pointer(&a.flags)) return rc;
  cudaError_t e = launch_tc_g128(a);
  return e == cudaSuccess ? W4A16_OK : cuda_fail(e, "w4a16_mm_g launch");
}

size_t w4a16_workspace_bytes(int N, int K) {
  if (N <= 0 || K <= 0 || K % kGroup || !tc_supported(N, K)) return 0;
  return tc_workspace_bytes();
}

int w4a16_mm_kernel(const w4a16_bf16* x, const uint32_t* Wq, const w4a16_bf16* scales, const w4a16_bf16* biases,
                    w4a16_bf16* y, int M, int N, int K, int kernel, void* stream) {
  return run_mm(x, Wq, scales, biases, y, M, N, K, kernel, stream);
}

int w4a16_mm_id(const w4a16_bf16* x, const uint32_t* Wq, const w4a16_bf16* scales, const w4a16_bf16* biases,
                const int32_t* ids, w4a16_bf16* y, int T, int N, int K, int E, void* stream) {
  return w4a16_mm_id_kernel(x, Wq, scales, biases, ids, y, T, N, K, E, W4A16_KERNEL_AUTO, stream);
}

int w4a16_mm_id_kernel(const w4a16_bf16* x, const uint32_t* Wq, const w4a16_bf16* scales,
                       const w4a16_bf16* biases, const int32_t* ids, w4a16_bf16* y, int T, int N, int K, int E,
                       int kernel, void* stream) {
  if (env().fault == kFaultValidate) return fail(W4A16_ERR_SHAPE, "injected validation fault (W4A16_FAULT)");
  if (T < 0 || T > kMaxDim) return fail(W4A16_ERR_EXPERTS, "T = %d must be in 0..2^30", T);
  if (E <= 0 || E > 65535) return fail(W4A16_ERR_EXPERTS, "E = %d must be in 1..65535", E);
  if (int rc = check_nk(N, K)) return rc;
  w4a16_plan plan;
  if (int rc = resolve_kernel(kernel, N, K, &plan)) return rc;
  if (K % 512 && plan.kernel == W4A16_KERNEL_TC_TILE)
    return fail(W4A16_ERR_KERNEL, "w4a16_mm_id with K %% 512 != 0 runs the persistent routed mode (K = %d)", K);
  if (T == 0) return W4A16_OK;
  if (!x || !Wq || !scales || !biases || !ids || !y) return fail(W4A16_ERR_NULL, "null tensor pointer");
  if (misaligned(x, 16) || misaligned(Wq, 16)) return fail(W4A16_ERR_ALIGN, "x and Wq must be 16-byte aligned");
  if (misaligned(scales, 8) || misaligned(biases, 8) || misaligned(y, 2) || misaligned(ids, 4))
    return fail(W4A16_ERR_ALIGN, "scales/biases must be 8-byte, y 2-byte and ids 4-byte aligned");
  if (plan.kernel == W4A16_KERNEL_VANILLA && T > 65535)
    return fail(W4A16_ERR_SHAPE, "the vanilla control kernel takes at most 65535 tokens");
  if (env().fault == kFaultLaunch) return fail(W4A16_ERR_CUDA, "injected launch fault (W4A16_FAULT)");
  LaunchArgs a{};
  a.x = x; a.Wq = Wq; a.S = scales; a.B = biases; a.y = y;
  a.N = N; a.K = K; a.ids = ids; a.T = T; a.E = E;
  a.stream = static_cast<cudaStream_t>(stream);
  a.pdl = env().pdl;
  a.tc_path = plan.kernel == W4A16_KERNEL_TC_STREAM ? 1 : plan.kernel == W4A16_KERNEL_TC_TILE ? 2 : 0;
  if (int rc = flag_pointer(&a.flags)) return rc;
  cudaError_t e = cudaSuccess;
  switch (plan.kernel) {
    case W4A16_KERNEL_SIMT: e = launch_simt_id(a, plan); break;
    case W4A16_KERNEL_TC:
    case W4A16_KERNEL_TC_STREAM:
    case W4A16_KERNEL_TC_TILE: e = launch_tc_id(a, plan); break;
    case W4A16_KERNEL_VANILLA: e = launch_vanilla_id(a, plan); break;
    default: return fail(W4A16_ERR_KERNEL, "kernel %d cannot run", plan.kernel);
  }
  if (e != cudaSuccess) return cuda_fail(e, "w4a16_mm_id launch");
  return W4A16_OK;
}

int w4a16_unpack(const uint32_t* Wq, uint8_t* q, int N, int K, void* stream) {
  if (N <= 0 || N > kMaxDim) return fail(W4A16_ERR_SHAPE, "N = %d must be in 1..2^30", N);
  if (K <= 0 || K > kMaxDim || K % 8) return fail(W4A16_ERR_SHAPE, "K = %d must be a positive multiple of 8", K);
  if (!Wq || !q) return fail(W4A16_ERR_NULL, "null tensor pointer");
  if (misaligned(Wq, 4) || misaligned(q, 8)) return fail(W4A16_ERR_ALIGN, "Wq must be 4-byte and q 8-byte aligned");
  cudaError_t e = launch_unpack(Wq, q, N, K, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4A16_OK : cuda_fail(e, "w4a16_unpack launch");
}

int w4a16_dequant(const uint32_t* Wq, const w4a16_bf16* scales, const w4a16_bf16* biases, float* w, int N, int K,
                  void* stream) {
  if (int rc = check_nk(N, K)) return rc;
  if (!Wq || !scales || !biases || !w) return fail(W4A16_ERR_NULL, "null tensor pointer");
  if (misaligned(Wq, 4) || misaligned(scales, 2) || misaligned(biases, 2) || misaligned(w, 16))
    return fail(W4A16_ERR_ALIGN, "Wq 4-byte, scales/biases 2-byte and w 16-byte alignment required");
  cudaError_t e = launch_dequant(Wq, scales, biases, w, N, K, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4A16_OK : cuda_fail(e, "w4a16_dequant launch");
}

int w4a16_expand_groups(const w4a16_bf16* src, w4a16_bf16* dst, int N, int K, int group, void* stream) {
  if (int rc = check_nk(N, K)) return rc;
  if (group < kGroup || group % kGroup || group > 4096 || K % group)
    return fail(W4A16_ERR_SHAPE, "group = %d must be a multiple of 64 that divides K = %d", group, K);
  if (!src || !dst) return fail(W4A16_ERR_NULL, "null tensor pointer");
  if (misaligned(src, 2) || misaligned(dst, 2)) return fail(W4A16_ERR_ALIGN, "src and dst must be 2-byte aligned");
  cudaError_t e = launch_expand_groups(src, dst, N, K, group, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4A16_OK : cuda_fail(e, "w4a16_expand_groups launch");
}

int w4a16_embed(const uint32_t* Wq, const w4a16_bf16* scales, const w4a16_bf16* biases, const int32_t* ids,
                w4a16_bf16* out, int T, int N, int K, void* stream) {
  if (env().fault == kFaultValidate) return fail(W4A16_ERR_SHAPE, "injected validation fault (W4A16_FAULT)");
  if (T < 0 || T > 65535) return fail(W4A16_ERR_SHAPE, "T = %d must be in 0..65535", T);
  if (int rc = check_nk(N, K)) return rc;
  if (T == 0) return W4A16_OK;
  if (!Wq || !scales || !biases || !ids || !out) return fail(W4A16_ERR_NULL, "null tensor pointer");
  if (misaligned(Wq, 4) || misaligned(scales, 2) || misaligned(biases, 2) || misaligned(ids, 4) || misaligned(out, 16))
    return fail(W4A16_ERR_ALIGN, "Wq and ids 4-byte, scales/biases 2-byte and out 16-byte alignment required");
  if (env().fault == kFaultLaunch) return fail(W4A16_ERR_CUDA, "injected launch fault (W4A16_FAULT)");
  int* flags = nullptr;
  if (int rc = flag_pointer(&flags)) return rc;
  cudaError_t e = launch_embed(Wq, scales, biases, ids, out, T, N, K, flags, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4A16_OK : cuda_fail(e, "w4a16_embed launch");
}

int w4a16_mm_noalloc(const w4a16_bf16* x, const uint32_t* Wq, const w4a16_bf16* scales, const w4a16_bf16* biases,
                     w4a16_bf16* y, int M, int N, int K, void* stream) {
  if (int rc = validate_mm(x, Wq, scales, biases, y, M, N, K)) return rc;
  if (!tc_supported(N, K))
    return fail(W4A16_ERR_KERNEL, "K = %d is past the tensor-core kernels' K %% 512 != 0 range", K);
  if (!tc_noalloc_fits(N, K))
    return fail(W4A16_ERR_SHAPE, "N = %d, K = %d needs more than the %zu-byte fixed scratch of w4a16_mm_noalloc", N, K,
                tc_noalloc_scratch_bytes());
  if (M == 0) return W4A16_OK;
  LaunchArgs a{};
  a.x = x; a.Wq = Wq; a.S = scales; a.B = biases; a.y = y;
  a.N = N; a.K = K;
  a.stream = static_cast<cudaStream_t>(stream);
  a.pdl = env().pdl;
  if (int rc = flag_pointer(&a.flags)) return rc;
  for (int row0 = 0; row0 < M; row0 += kMaxChunk) {
    a.row0 = row0;
    a.M = (M - row0 < kMaxChunk) ? M - row0 : kMaxChunk;
    cudaError_t e = launch_tc_noalloc(a);
    if (e == cudaErrorInvalidValue) return fail(W4A16_ERR_SHAPE, "shape exceeds the fixed scratch of w4a16_mm_noalloc");
    if (e != cudaSuccess) return cuda_fail(e, "w4a16_mm_noalloc launch");
  }
  return W4A16_OK;
}

int w4a16_mm_argmax(const w4a16_bf16* x, const uint32_t* Wq, const w4a16_bf16* scales, const w4a16_bf16* biases,
                    int32_t* idx, w4a16_bf16* val, int M, int N, int K, void* workspace, size_t workspace_bytes,
                    void* stream) {
  if (env().fault == kFaultValidate) return fail(W4A16_ERR_SHAPE, "injected validation fault (W4A16_FAULT)");
  if (int rc = validate_mm(x, Wq, scales, biases, idx, M, N, K)) return rc;
  if (M == 0) return W4A16_OK;
  if (!workspace) return fail(W4A16_ERR_NULL, "w4a16_mm_argmax needs a workspace (w4a16_workspace_bytes)");
  if (int rc = check_workspace(workspace, workspace_bytes)) return rc;
  if (misaligned(idx, 4) || misaligned(val, 2)) return fail(W4A16_ERR_ALIGN, "idx must be 4-byte and val 2-byte aligned");
  if (K % 512)
    return fail(W4A16_ERR_KERNEL, "w4a16_mm_argmax runs the tensor-core kernel, which needs K %% 512 == 0 (K = %d)", K);
  if (env().fault == kFaultLaunch) return fail(W4A16_ERR_CUDA, "injected launch fault (W4A16_FAULT)");
  LaunchArgs a{};
  a.x = x; a.Wq = Wq; a.S = scales; a.B = biases; a.y = nullptr;
  a.N = N; a.K = K;
  a.stream = static_cast<cudaStream_t>(stream);
  a.pdl = env().pdl;
  a.tc_path = 1;
  a.ws = workspace;
  a.ws_bytes = workspace_bytes;
  if (int rc = flag_pointer(&a.flags)) return rc;
  for (int row0 = 0; row0 < M; row0 += kMaxChunk) {
    a.row0 = row0;
    a.M = (M - row0 < kMaxChunk) ? M - row0 : kMaxChunk;
    cudaError_t e = launch_tc_argmax(a, idx, val);
    if (e == cudaErrorInvalidValue) return fail(W4A16_ERR_SHAPE, "N = %d, K = %d exceeds the persistent kernel's workspace", N, K);
    if (e != cudaSuccess) return cuda_fail(e, "w4a16_mm_argmax launch");
  }
  return W4A16_OK;
}

int w4a16_mm_group(const w4a16_mm_item* items, int count, int M, int K, void* stream) {
  if (env().fault == kFaultValidate) return fail(W4A16_ERR_SHAPE, "injected validation fault (W4A16_FAULT)");
  if (count < 1 || count > W4A16_MAX_GROUP)
    return fail(W4A16_ERR_SHAPE, "count = %d must be in 1..%d", count, W4A16_MAX_GROUP);
  if (!items) return fail(W4A16_ERR_NULL, "null item array");
  int Ns[W4A16_MAX_GROUP];
  for (int i = 0; i < count; ++i) {
    const w4a16_mm_item& it = items[i];
    if (int rc = validate_mm(it.x, it.Wq, it.scales, it.biases, it.y, M, it.N, K)) return rc;
    Ns[i] = it.N;
  }
  if (M == 0) return W4A16_OK;
  if (env().force_kernel != W4A16_KERNEL_AUTO || !tc_group_supported(Ns, count, K)) {
    for (int i = 0; i < count; ++i) {
      const w4a16_mm_item& it = items[i];
      if (int rc = run_mm(it.x, it.Wq, it.scales, it.biases, it.y, M, it.N, K, W4A16_KERNEL_AUTO, stream)) return rc;
    }
    return W4A16_OK;
  }
  if (env().fault == kFaultLaunch) return fail(W4A16_ERR_CUDA, "injected launch fault (W4A16_FAULT)");
  int* flags = nullptr;
  if (int rc = flag_pointer(&flags)) return rc;
  GroupItem g[W4A16_MAX_GROUP];
  for (int i = 0; i < count; ++i)
    g[i] = GroupItem{items[i].x, items[i].Wq, items[i].scales, items[i].biases, items[i].y, items[i].N};
  cudaError_t e = launch_tc_group(g, count, M, 0, K, env().pdl, flags, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "w4a16_mm_group launch");
  return W4A16_OK;
}

int w4a16_get_plan(int N, int K, int kernel, w4a16_plan* out) {
  if (!out) return fail(W4A16_ERR_NULL, "null plan pointer");
  if (int rc = check_nk(N, K)) return rc;
  return resolve_kernel(kernel, N, K, out);
}

int w4a16_device_status(void* stream, int* flags) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int* p = nullptr;
  if (int rc = flag_pointer(&p)) return rc;
  int v = 0;
  e = cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read device flags");
  if (flags) *flags = v;
  if (v) {
    const int zero = 0;
    e = cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clear device flags");
    return fail(W4A16_ERR_DEVICE, "a kernel reported bad input (flags 0x%x)", v);
  }
  return W4A16_OK;
}

// ---- STQ1_0 (include/stq1.h) ----------------------------------------------------

size_t stq1_packed_bytes(int N, int K) { return stq1_packed_size(N, K); }

int stq1_get_plan(int N, int K, stq1_plan* out) {
  if (!out) return fail(W4A16_ERR_NULL, "null plan pointer");
  if (!stq1_shape_ok(N, K))
    return fail(W4A16_ERR_SHAPE, "N = %d must be >= 1 and K = %d a multiple of 256 in 256..%d", N, K, STQ1_MAX_K);
  Stq1Plan p;
  stq1_make_plan(N, K, &p);
  out->ksplit = p.ks;
  out->blocks_per_slice = p.bps;
  out->rows_per_pass = p.xcap;
  return W4A16_OK;
}

int stq1_pack(const uint8_t* blocks, uint8_t* packed, int N, int K, void* stream) {
  if (!stq1_shape_ok(N, K))
    return fail(W4A16_ERR_SHAPE, "N = %d must be >= 1 and K = %d a multiple of 256 in 256..%d", N, K, STQ1_MAX_K);
  if (!blocks || !packed) return fail(W4A16_ERR_NULL, "null tensor pointer");
  if (misaligned(blocks, 2) || misaligned(packed, 16))
    return fail(W4A16_ERR_ALIGN, "blocks must be 2-byte and packed 16-byte aligned");
  cudaError_t e = launch_stq1_pack(blocks, packed, N, K, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4A16_OK : cuda_fail(e, "stq1_pack launch");
}

int stq1_mm(const float* x, const uint8_t* packed, float* y, int M, int N, int K, void* stream) {
  if (env().fault == kFaultValidate) return fail(W4A16_ERR_SHAPE, "injected validation fault (W4A16_FAULT)");
  if (M < 0 || M > kMaxDim) return fail(W4A16_ERR_SHAPE, "M = %d must be in 0..2^30", M);
  if (!stq1_shape_ok(N, K) || N > kMaxDim)
    return fail(W4A16_ERR_SHAPE, "N = %d must be in 1..2^30 and K = %d a multiple of 256 in 256..%d", N, K,
                STQ1_MAX_K);
  if (M == 0) return W4A16_OK;
  if (!x || !packed || !y) return fail(W4A16_ERR_NULL, "null tensor pointer");
  if (misaligned(x, 16) || misaligned(packed, 16) || misaligned(y, 4))
    return fail(W4A16_ERR_ALIGN, "x and packed must be 16-byte and y 4-byte aligned");
  if (env().fault == kFaultLaunch) return fail(W4A16_ERR_CUDA, "injected launch fault (W4A16_FAULT)");
  int* flags = nullptr;
  if (int rc = flag_pointer(&flags)) return rc;
  Stq1Plan pl;
  stq1_make_plan(N, K, &pl);
  for (int row0 = 0; row0 < M; row0 += pl.xcap) {
    const int rows = M - row0 < pl.xcap ? M - row0 : pl.xcap;
    cudaError_t e =
        launch_stq1_mm(x, packed, y, rows, row0, N, K, flags, env().pdl, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "stq1_mm launch");
  }
  return W4A16_OK;
}

int stq1_mm_id(const float* x, const uint8_t* packed, const int32_t* ids, float* y, int T, int N, int K, int E,
               void* stream) {
  if (env().fault == kFaultValidate) return fail(W4A16_ERR_SHAPE, "injected validation fault (W4A16_FAULT)");
  if (T < 0 || T > kMaxDim) return fail(W4A16_ERR_EXPERTS, "T = %d must be in 0..2^30", T);
  if (E <= 0 || E > 65535) return fail(W4A16_ERR_EXPERTS, "E = %d must be in 1..65535", E);
  if (!stq1_shape_ok(N, K) || N > kMaxDim)
    return fail(W4A16_ERR_SHAPE, "N = %d must be in 1..2^30 and K = %d a multiple of 256 in 256..%d", N, K,
                STQ1_MAX_K);
  if (T == 0) return W4A16_OK;
  if (!x || !packed || !ids || !y) return fail(W4A16_ERR_NULL, "null tensor pointer");
  if (misaligned(x, 16) || misaligned(packed, 16) || misaligned(y, 4) || misaligned(ids, 4))
    return fail(W4A16_ERR_ALIGN, "x and packed must be 16-byte, y and ids 4-byte aligned");
  if (env().fault == kFaultLaunch) return fail(W4A16_ERR_CUDA, "injected launch fault (W4A16_FAULT)");
  int* flags = nullptr;
  if (int rc = flag_pointer(&flags)) return rc;
  cudaError_t e =
      launch_stq1_mm_id(x, packed, ids, y, T, N, K, E, flags, env().pdl, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4A16_OK : cuda_fail(e, "stq1_mm_id launch");
}

int stq1_get_rows(const uint8_t* packed, const int32_t* ids, float* out, int T, int N, int K, void* stream) {
  if (T < 0 || T > kMaxDim) return fail(W4A16_ERR_SHAPE, "T = %d must be in 0..2^30", T);
  if (!stq1_shape_ok(N, K) || N > kMaxDim)
    return fail(W4A16_ERR_SHAPE, "N = %d must be in 1..2^30 and K = %d a multiple of 256 in 256..%d", N, K,
                STQ1_MAX_K);
  if (T == 0) return W4A16_OK;
  if (!packed || !ids || !out) return fail(W4A16_ERR_NULL, "null tensor pointer");
  if (misaligned(packed, 16) || misaligned(ids, 4) || misaligned(out, 4))
    return fail(W4A16_ERR_ALIGN, "packed must be 16-byte, ids and out 4-byte aligned");
  int* flags = nullptr;
  if (int rc = flag_pointer(&flags)) return rc;
  cudaError_t e = launch_stq1_get_rows(packed, ids, out, T, N, K, flags, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4A16_OK : cuda_fail(e, "stq1_get_rows launch");
}

const char* w4a16_last_error(void) { return g_last_error.c_str(); }

const char* w4a16_version(void) { return "w4a16 0.1.0 (sm_103a)"; }

void w4a16_debug_reload_env(void) {
  std::lock_guard<std::mutex> lk(g_env_mu);
  load_env_locked();
}

}  // extern "C"

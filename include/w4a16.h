/*
 * w4a16.h -- C ABI of libw4a16.so: weight-only 4-bit, group-64 affine
 * quantized matmul (W4A16) for skinny activations on GB300 (sm_103a).
 *
 * Citations (page titles; sections in quotes):
 *   [W2D2] tiny-llm book, "Week 2 Day 2: Keep W4 Packed"
 *   [G4MK] "Gemma 4 E4B & E2B -- single-launch Metal megakernels + lossless
 *          speculative decoding" (RESMP-DEV model card)
 *   [HY4]  "Hy4-preview Metal kernels for llama.cpp"
 *
 * The operation ([W2D2 "Mathematical Formulation", C = A B^T, and
 * "Reconstruct a Stored Group", w^ = q s + b]):
 *
 *   q[n,k] = (Wq[n][k/8] >> 4*(k%8)) & 0xF            (low nibble first,
 *                                                      [W2D2 "Packed Storage Layout"])
 *   y[m,n] = bf16( sum_k x[m,k] * (q[n,k]*scales[n][k/64] + biases[n][k/64]) )
 *
 * with the group size fixed at 64 ([G4MK "Usage": 4-bit weights at group
 * size 64; the dequant path assumes it]).  The page writes A (M x N), B
 * (K x N), C (M x K) with the reduction over N; this header uses
 * x[M][K], Wq[N][K/8], y[M][N] with the reduction over K.
 *
 * Layout.  Every tensor is dense and row-major with no strides (the
 * row-contiguous contract of [W2D2 "Tune the SIMD Schedule"]):
 *   x       bf16 [M][K]        activations
 *   Wq      u32  [N][K/8]      eight 4-bit codes per word, code k%8 in bits 4*(k%8)..+3
 *   scales  bf16 [N][K/64]     signed; used as stored ([W2D2 "Reconstruct a Stored Group"])
 *   biases  bf16 [N][K/64]
 *   y       bf16 [M][N]        round-to-nearest-even of the fp32 accumulation
 * bf16 values are passed as raw 16-bit patterns (w4a16_bf16).
 *
 * Batch invariance ([G4MK "What it does" and "Implementation notes": the
 * verify GEMM is arithmetic-identical to the sequential GEMV, batch equals
 * sequential bitwise]).  The kernel and its reduction order are chosen from
 * (N, K) only, never from M, so row m of any call equals, bit for bit, the
 * M = 1 call on x[m].  Calls with M > 8 take the rows eight at a time
 * through the same arithmetic (the tile kernel in one launch over resident
 * weights, the other kernels one launch per chunk).  w4a16_mm_id rows equal
 * w4a16_mm on the selected expert, bit for bit.
 *
 * Ownership and synchronisation.  All tensor pointers are DEVICE pointers
 * owned by the caller, and the library allocates no device memory: no
 * compute call calls cudaMalloc or keeps per-stream state, so every call
 * (its first one included) may be captured into a CUDA graph.  `stream` is
 * a cudaStream_t (NULL = legacy default stream).  Compute calls only
 * enqueue work: they return before the GPU is done and never synchronise,
 * except w4a16_device_status.
 *
 * Overlapped launches.  The tensor-core kernels are launched as programmatic
 * dependents: a call may start while the previous kernel on its stream is
 * still running, and (unless the environment sets W4A16_PDL=1 or 0) it
 * requests its first weight tiles before it waits for that kernel.  It reads
 * activations and ids, and writes outputs, only after the wait.  So the
 * weights (Wq, scales, biases) must not be written by work still pending on
 * the same stream: finish writing them (synchronise, or make the stream wait
 * on an event recorded after the writes) before the first call that reads
 * them.  W4A16_PDL=1 keeps the overlap without the early fetch; 0 turns both
 * off.
 *
 * Workspace (optional for w4a16_mm_ws, required by w4a16_mm_argmax).  A
 * caller-owned block of device memory of w4a16_workspace_bytes(N, K) bytes
 * (4.78 MiB, the same for every shape; 256-byte aligned) in which the
 * persistent tensor-core grid keeps a unit counter shared by all its CTAs,
 * the fp32 slice sums of a K split across SMs and the argmax keys.  The
 * caller zeroes it once before its first use (cudaMemsetAsync); every call
 * that completes leaves it zeroed again, and after w4a16_device_status
 * reports W4A16_DEVICE_TIMEOUT it must be zeroed again.  Calls that share a
 * workspace must not overlap on the GPU (one stream, or ordered by events).
 * Without a workspace (w4a16_mm) the same arithmetic runs in shapes that
 * need none: work units are dealt inside each CTA, and a K split across SMs
 * becomes a cluster of CTAs adding the slice sums in distributed shared
 * memory or, where a cluster cannot hold a tile's K range, whole-K units
 * that fold the slice sums in registers.  The results are the same bits
 * either way.
 *
 * Alignment.  x and Wq must be 16-byte aligned (their rows then are too,
 * because K % 64 == 0); scales and biases 8-byte aligned; y 2-byte; ids
 * 4-byte.
 *
 * Errors ("fail closed": arguments are checked on the host before any
 * launch, and a rejected call writes nothing, after [W2D2 "Task 2": validate
 * inputs and reject unsupported evaluation explicitly]).  Every call returns
 * a w4a16_status; the message of the last failure on the calling host
 * thread is kept for w4a16_last_error().
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t w4a16_bf16; /* raw bfloat16 bits */

typedef enum {
  W4A16_OK = 0,
  W4A16_ERR_NULL = -1,      /* a required pointer is NULL */
  W4A16_ERR_SHAPE = -2,     /* K <= 0, K % 64 != 0, N <= 0, M < 0, or too large */
  W4A16_ERR_ALIGN = -3,     /* x / Wq not 16-byte aligned, or another pointer misaligned */
  W4A16_ERR_EXPERTS = -4,   /* E <= 0 or T < 0 */
  W4A16_ERR_CUDA = -5,      /* a CUDA call or launch failed; see w4a16_last_error() */
  W4A16_ERR_KERNEL = -6,    /* unknown kernel selector */
  W4A16_ERR_DEVICE = -7     /* w4a16_device_status: a kernel reported bad input */
} w4a16_status;

/* Kernel families (all compute the operation above). */
typedef enum {
  W4A16_KERNEL_AUTO = 0,    /* the dispatcher's choice for (N, K) */
  W4A16_KERNEL_SIMT = 1,    /* CUDA-core kernel: fp32 FMA, warp-shuffle split-K */
  W4A16_KERNEL_TC = 2,      /* tensor-core kernel: TMA-fed bf16 MMA on codes, fp32 group
                               rescale.  K % 512 == 0 runs as one of the launch shapes
                               below, chosen from (N, K, M), all with identical bits.
                               K % 512 != 0 runs padded to whole 512-code stages (the
                               padding groups add exactly +0) on the persistent and tile
                               shapes, whose work units bring their scale and bias rows
                               by bulk copy; up to K = 5952, where those rows fit in
                               shared memory next to eight activation rows (larger:
                               W4A16_ERR_KERNEL; the dispatcher takes the CUDA-core
                               family there) */
  W4A16_KERNEL_VANILLA = 3, /* debug control: one thread per output, no sharing */
  W4A16_KERNEL_TC_STREAM = 4, /* tensor-core kernel, persistent grid: work units dealt to
                                 warps from a counter (in the CTA without a workspace);
                                 without a workspace a split K runs as whole-K units.
                                 w4a16_mm_id: T <= 32 its routed mode, more tokens a grid
                                 of tile x expert CTAs */
  W4A16_KERNEL_TC_TILE = 5, /* tensor-core kernel, one CTA per 16-row tile holding the
                               tile's whole K range; needs that to fit in shared memory
                               (otherwise W4A16_ERR_KERNEL); w4a16_mm_id with K % 512 != 0
                               runs the persistent routed mode only (W4A16_ERR_KERNEL) */
  W4A16_KERNEL_TC_PREFILL = 6 /* tensor-core kernel for many rows: each 64-code group of a
                                 128-row tile expanded once to bf16 in shared memory, then
                                 tcgen05.mma over up to 128 activation rows into tensor
                                 memory; the default for M > 32 where the family applies;
                                 needs K % 512 == 0 (otherwise W4A16_ERR_KERNEL; with
                                 K % 512 != 0 the dispatcher runs M > 32 on the
                                 persistent shape, eight rows a launch) */
} w4a16_kernel;

/* y[M][N] = x[M][K] W^T.  M == 0 is a successful no-op.  The kernel family
 * is the dispatcher's choice for (N, K) unless the environment variable
 * W4A16_FORCE_KERNEL names one (simt, tc, vanilla).  Uses no workspace. */
int w4a16_mm(const w4a16_bf16* x, const uint32_t* Wq, const w4a16_bf16* scales,
             const w4a16_bf16* biases, w4a16_bf16* y, int M, int N, int K, void* stream);

/* w4a16_mm with the caller's workspace (see "Workspace" above; NULL runs
 * w4a16_mm).  With one, the persistent grid deals its units from one
 * counter over all SMs and splits K across SMs where the canonical slicing
 * has several slices (w4a16_get_plan: workspace_bytes > 0 and ksplit > 1):
 * the fastest launch shape for large matrices.  Results equal w4a16_mm bit
 * for bit.  A workspace smaller than w4a16_workspace_bytes(N, K) is
 * W4A16_ERR_SHAPE, one not 256-byte aligned W4A16_ERR_ALIGN. */
int w4a16_mm_ws(const w4a16_bf16* x, const uint32_t* Wq, const w4a16_bf16* scales,
                const w4a16_bf16* biases, w4a16_bf16* y, int M, int N, int K, void* workspace,
                size_t workspace_bytes, void* stream);

/* Bytes of workspace the tensor-core family can use for (N, K): 0 when it
 * does not apply (an invalid shape, or K % 512 != 0 past K = 5952),
 * otherwise a fixed 5,013,504 bytes (32 KiB of counters + 4864 KiB of fp32
 * partials; with K % 512 != 0 only the unit counter is used). */
size_t w4a16_workspace_bytes(int N, int K);

/* w4a16_mm with an explicit kernel family (for A/B comparisons and tests). */
int w4a16_mm_kernel(const w4a16_bf16* x, const uint32_t* Wq, const w4a16_bf16* scales,
                    const w4a16_bf16* biases, w4a16_bf16* y, int M, int N, int K,
                    int kernel, void* stream);

/* w4a16_mm for callers that must not allocate device memory (no counterpart
 * on the pages; this is a deployment variant, not part of the method).
 * Who needs it: code running inside an engine that reserved all device
 * memory at start-up and hands out nothing more, processes under a hard
 * device-memory cap where a late cudaMalloc could fail mid-service, and
 * deployments that forbid allocation after initialisation.  Like w4a16_mm
 * it never calls cudaMalloc, cudaFree or any allocating routine; unlike
 * w4a16_mm it always runs the persistent grid with a K split across SMs,
 * its workspace being a fixed array inside the library.
 *
 * It runs the same tensor-core kernel with the same arithmetic, so its
 * results equal w4a16_mm's bit for bit.  Its split-K scratch is one fixed
 * 5,013,504-byte device array inside the library (32 KiB of tile counters +
 * 4864 KiB of fp32 partials), which every GPU that loads the library holds
 * until the process exits; every (N, K) with K % 512 == 0 fits in it, and a
 * shape that would not is rejected with W4A16_ERR_SHAPE.  K % 512 != 0 runs
 * in whole-K units without scratch, up to K = 5952 (larger:
 * W4A16_ERR_KERNEL).
 *
 * The first call on a device looks up the array's device address and sets
 * the kernel's shared-memory limit; make that first call before any CUDA
 * graph capture.  Under CUDA's default lazy module loading the array itself
 * is committed on the device when the library's kernels are first loaded,
 * which for a process that calls nothing else is that first call: a caller
 * under a hard memory cap makes it at start-up (or sets
 * CUDA_MODULE_LOADING=EAGER), so that nothing is committed mid-service.  All calls share the one array and it keeps the last
 * call's contents: each call clears the counters it uses (a memset on
 * `stream`) before its kernel.  Calls whose executions overlap on the GPU
 * (different streams, or graphs replayed concurrently) race on the array;
 * keep them ordered. */
int w4a16_mm_noalloc(const w4a16_bf16* x, const uint32_t* Wq, const w4a16_bf16* scales,
                     const w4a16_bf16* biases, w4a16_bf16* y, int M, int N, int K, void* stream);

/* Fused argmax over the outputs (greedy decoding on a tied LM head; the
 * drafter of [G4MK] "Implementation notes" runs its head with an in-kernel
 * argmax):
 *   idx[m] = argmax_n bf16(y[m][n]),  val[m] = bf16(y[m][idx[m]])
 * where y is exactly what w4a16_mm computes (the same canonical arithmetic,
 * so idx is the argmax of w4a16_mm's rows bit for bit); y is never written.
 * Ties go to the smallest n; a NaN output ranks above every number and
 * -0 just below +0.
 * idx int32 [M] (4-byte aligned) and val bf16 [M] (may be NULL) are device
 * pointers.  Runs the persistent tensor-core kernel: needs K % 512 == 0
 * (otherwise W4A16_ERR_KERNEL).  The CTAs merge their keys in the caller's
 * workspace (see "Workspace" above; NULL is W4A16_ERR_NULL, too small
 * W4A16_ERR_SHAPE); other errors as w4a16_mm. */
int w4a16_mm_argmax(const w4a16_bf16* x, const uint32_t* Wq, const w4a16_bf16* scales,
                    const w4a16_bf16* biases, int32_t* idx, w4a16_bf16* val, int M, int N, int K,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Grouped projections: several independent w4a16_mm calls that share K and
 * M, in one launch where that pays (a decoder layer's q/k/v projections read
 * the same activations, as do gate/up; launching them together saves the
 * per-launch latency that dominates decode-sized matmuls).  No counterpart
 * on the pages; each item is exactly the operation of w4a16_mm above.
 *
 * `items` is a HOST array of `count` (1..W4A16_MAX_GROUP) descriptors; the
 * pointers inside are device pointers with w4a16_mm's layout and alignment
 * (x [M][K], Wq [N][K/8], scales/biases [N][K/64], y [M][N]).  Items are
 * independent: no item's y may overlap any other item's operands or y.  Row
 * m of every item's y equals, bit for bit, w4a16_mm on that item.  When the
 * shapes do not allow one launch (K % 512 != 0, or an item too large for the
 * tile launch shape) the items run as consecutive w4a16_mm calls.  Errors
 * are those of w4a16_mm, checked for every item before anything is
 * launched; count outside 1..W4A16_MAX_GROUP is W4A16_ERR_SHAPE. */
#define W4A16_MAX_GROUP 8

typedef struct {
  const w4a16_bf16* x;      /* [M][K] activations of this item */
  const uint32_t* Wq;       /* [N][K/8] packed codes */
  const w4a16_bf16* scales; /* [N][K/64] */
  const w4a16_bf16* biases; /* [N][K/64] */
  w4a16_bf16* y;            /* [M][N] output */
  int N;                    /* output columns of this item */
} w4a16_mm_item;

int w4a16_mm_group(const w4a16_mm_item* items, int count, int M, int K, void* stream);

/* Routed experts, top-1 (the W4A16 analogue of llama.cpp's mul_mat_id named
 * in [HY4] "What was missing and what this adds"):
 *   y[t][n] = sum_k x[t][k] * w_{ids[t]}[n][k]
 * Wq is u32 [E][N][K/8], scales/biases bf16 [E][N][K/64], ids int32 [T] on
 * the DEVICE, y bf16 [T][N].  The tokens of an expert are taken in chunks
 * of up to eight; experts no token selects are not read.  With T <= 32 every
 * chunk streams its expert's weights once (the chunks run side by side, the
 * units of all of them dealt over one persistent grid); with more tokens a
 * CTA holds a tile of an expert's weights in shared memory while all its
 * chunks stream through.  An id outside 0..E-1 cannot be checked on the
 * host without a synchronisation: its row of y is written as zeros and the
 * sticky device flag W4A16_DEVICE_BAD_ID is raised (see w4a16_device_status).
 * T == 0 is a successful no-op. */
int w4a16_mm_id(const w4a16_bf16* x, const uint32_t* Wq, const w4a16_bf16* scales,
                const w4a16_bf16* biases, const int32_t* ids, w4a16_bf16* y,
                int T, int N, int K, int E, void* stream);

/* w4a16_mm_id with an explicit kernel family. */
int w4a16_mm_id_kernel(const w4a16_bf16* x, const uint32_t* Wq, const w4a16_bf16* scales,
                       const w4a16_bf16* biases, const int32_t* ids, w4a16_bf16* y,
                       int T, int N, int K, int E, int kernel, void* stream);

/* The operation with the group size as an argument (the tiny-llm book
 * quantizes with 128 codes per scale and bias, [W2D2] "Packed Storage
 * Layout"): scales and biases are bf16 [N][K/group],
 *   y[m,n] = bf16( sum_k x[m,k] * (q[n,k]*scales[n][k/group] + biases[n][k/group]) ).
 * group 64 is w4a16_mm_ws.  group 128 reads the tables as they are, 0.53125
 * bytes per weight instead of the 0.5625 of an expansion to group 64
 * ([W2D2] "Revisit the Decode Roofline"), on the persistent tensor-core grid
 * in whole-K work units: K % 512 == 0 and K <= 8192 (other K:
 * W4A16_ERR_SHAPE; expand with w4a16_expand_groups instead), scales and
 * biases 16-byte aligned (W4A16_ERR_ALIGN).  Every 64-group is rescaled with
 * its 128-group's pair, so y equals, bit for bit, the group-64 entry points on
 * the expanded tables, and row m of any call equals the M = 1 call on x[m].
 * The workspace (may be NULL) only deals the work units; otherwise as
 * w4a16_mm_ws. */
int w4a16_mm_g(const w4a16_bf16* x, const uint32_t* Wq, const w4a16_bf16* scales,
               const w4a16_bf16* biases, w4a16_bf16* y, int M, int N, int K, int group, void* workspace,
               size_t workspace_bytes, void* stream);

/* Tables quantized with a larger group (the tiny-llm book quantizes with 128
 * codes per scale and bias, [W2D2] "Packed Storage Layout"): dst[n][j] =
 * src[n][j / (group / 64)], the scales (or biases) of every group repeated
 * over its 64-code parts, bf16 [N][K/group] -> bf16 [N][K/64] on the device.
 * With the expanded scales and biases the group-64 entry points compute
 * q * s + b with each weight's own s and b, i.e. the larger-group matmul
 * (the parameters then cost 4/64 instead of 4/group bytes per weight).
 * group: a multiple of 64 that divides K, at most 4096.  Call it once when
 * the weights are loaded. */
int w4a16_expand_groups(const w4a16_bf16* src, w4a16_bf16* dst, int N, int K, int group, void* stream);

/* Quantized embedding rows (the row lookup of [W2D2] "Task 1: Implement
 * Quantized Linear and Embedding": gather the selected packed rows, unpack,
 * q * scale + bias; the table stays packed):
 *   out[t][k] = bf16(fp32 fma(q[ids[t]][k], s, b))   for t < T, k < K
 * with the single-rounding fp32 fma of w4a16_dequant and round-to-nearest-
 * even to bf16.  Wq u32 [N][K/8], scales/biases bf16 [N][K/64] (the table:
 * N rows of width K), ids int32 [T] and out bf16 [T][K] on the DEVICE (out
 * 16-byte aligned).  An id outside 0..N-1 gives a zero row and raises
 * W4A16_DEVICE_BAD_ID.  T in 0..65535; T == 0 is a successful no-op. */
int w4a16_embed(const uint32_t* Wq, const w4a16_bf16* scales, const w4a16_bf16* biases, const int32_t* ids,
                w4a16_bf16* out, int T, int N, int K, void* stream);

/* Debug: q[N][K] (one byte per code) from Wq[N][K/8].  Bit-exact
 * ([W2D2 "Packed Storage Layout"]). */
int w4a16_unpack(const uint32_t* Wq, uint8_t* q, int N, int K, void* stream);

/* Debug: w[N][K] = fp32 fma(q, s, b) (one rounding), K % 64 == 0
 * ([W2D2 "Reconstruct a Stored Group"]). */
int w4a16_dequant(const uint32_t* Wq, const w4a16_bf16* scales, const w4a16_bf16* biases,
                  float* w, int N, int K, void* stream);

/* The dispatcher's decision for a shape.  `ksplit` and `slice_k` fix the
 * reduction order of every output row: K is cut into `ksplit` consecutive
 * slices of `slice_k` codes (the last one may be shorter); each slice is
 * reduced on its own and the slice sums are added in slice order.  Both
 * depend on (N, K) only, never on M.  The other fields describe the launch
 * of one chunk of at most eight activation rows on this device (152 SMs are
 * assumed when no GPU is present), for w4a16_mm_ws given a workspace. */
typedef struct {
  int kernel;        /* w4a16_kernel actually used */
  int ksplit;        /* K-slices per output row */
  int slice_k;       /* codes per K-slice */
  int rows_per_tile; /* output rows of one work unit */
  int units;         /* work units (row tile x K-slice) of one chunk */
  int threads;       /* threads per CTA */
  int grid_x;        /* CTAs per chunk */
  int smem_bytes;    /* dynamic shared memory per CTA (M = 1) */
  int workspace_bytes; /* workspace this launch shape uses when one is given (w4a16_mm_ws), else 0 */
} w4a16_plan;

int w4a16_get_plan(int N, int K, int kernel, w4a16_plan* out);

/* Sticky device-side error flags, raised by kernels instead of trapping. */
#define W4A16_DEVICE_BAD_ID 1   /* mm_id: an expert id outside 0..E-1 */
#define W4A16_DEVICE_TIMEOUT 2  /* a bounded wait on an asynchronous copy gave up */

/* Synchronises `stream`, reads and clears the device flags of the current
 * device.  Returns W4A16_OK when no flag was set, W4A16_ERR_DEVICE when one
 * was (flags stored in *flags if non-NULL), W4A16_ERR_CUDA on a CUDA error. */
int w4a16_device_status(void* stream, int* flags);

/* Message of the last failed call on this host thread ("" if none). */
const char* w4a16_last_error(void);

/* Debug: re-read the environment switches W4A16_FAULT (validate | launch:
 * every compute call then fails with that error before launching anything;
 * wait: in every persistent-grid launch of w4a16_mm one stage of one warp
 * expects 16 bytes more than its copies deliver, so that warp's bounded wait
 * gives up, raises W4A16_DEVICE_TIMEOUT and leaves its rows unwritten; every
 * copy still lands, so nothing is in flight when the kernel exits) and
 * W4A16_FORCE_KERNEL (simt | tc | vanilla).  They are read once, at the
 * first call, otherwise. */
void w4a16_debug_reload_env(void);

/* Library version string. */
const char* w4a16_version(void);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */

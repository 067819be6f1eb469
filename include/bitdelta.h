/*
 * bitdelta.h -- C ABI of the BitDelta GB300 (sm_103a) library.
 *
 * The method is the one on the web page "BitDelta: serving 14 Zen models from
 * one GPU cluster" (Hanzo blog, 2026-02-28):
 *   section "The mathematical foundation": delta = W_ft - W_base, one scale
 *     alpha = mean|delta| per matrix, and one sign bit per weight, so that
 *     W_ft ~ W_base + alpha * sign(delta);
 *   section "Serving architecture": many fine-tuned variants share one
 *     resident base; a fused kernel reads the base weights and the packed
 *     delta bits together and never writes W_eff to HBM (the conceptual
 *     fused_bitdelta_linear listing: reconstruct, then linear).  The decode
 *     paths here never write W_eff; the prefill path writes it, once per
 *     present variant and into the caller's workspace, when the batch has at
 *     least 2048 tokens per present variant (see BD_PATH_PREFILL_TC);
 *   section "Infrastructure details": sign bits packed 8 per byte (a
 *     4096 x 4096 weight packs to 4096 x 512 bytes), alpha stored as f32.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers.  Every array argument is a DEVICE pointer unless its comment says
 *   HOST.  The caller owns every buffer (inputs, outputs and workspace); the
 *   library allocates nothing and keeps no per-call state.
 * Layouts.  Matrices are row-major with leading dimension equal to their
 *   column count.  W_base, W_ft are [N, K] (N = d_out rows, K = d_in columns);
 *   activations x are [M, K]; outputs y are [M, N].
 * Packed sign bits.  [N, K/32] little-endian u32 words: bit j of word w in row
 *   n is column 32*w + j; the bit is 1 when W_ft >= W_base (so a zero delta,
 *   of either sign, counts as +1) and 0 otherwise.  Byte for byte this is an
 *   int8/uint8 [N, K/8] matrix whose bit i of byte b is column 8*b + i.
 * Streams.  `stream` is a cudaStream_t passed as void*; NULL is the legacy
 *   default stream.  Every call is asynchronous on it: it validates its
 *   arguments on the host, enqueues kernels and returns.
 * Errors.  Argument errors are found on the host before anything is
 *   enqueued and returned directly (nothing is launched).  Errors only the
 *   device can see (a variant id out of range, a bounded wait that ran out)
 *   are OR-ed into a status word at the start of the workspace; read it with
 *   bitdelta_device_status().  A launch failure returns BD_ERR_CUDA.
 * Alignment.  Every device array must start on a 16-byte boundary, except
 *   alpha arrays and variant_ids (4 bytes).
 * Concurrency.  Calls are reentrant; calls that run at the same time on the
 *   GPU must use distinct workspaces.
 */
#ifndef BITDELTA_H
#define BITDELTA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BITDELTA_ABI_VERSION 1
#define BITDELTA_MAX_VARIANTS 64

typedef enum {
    BD_OK = 0,
    BD_ERR_NULL = 1,        /* a required pointer is NULL */
    BD_ERR_ALIGN = 2,       /* a pointer is not 16-byte (or 4-byte) aligned */
    BD_ERR_SHAPE = 3,       /* bad size: N, K < 1, K % 32 != 0, M < 0, V out of range */
    BD_ERR_DTYPE = 4,       /* unsupported dtype code */
    BD_ERR_VARIANT = 5,     /* device: a variant id outside [-1, V) */
    BD_ERR_WORKSPACE = 6,   /* workspace NULL or smaller than the *_workspace() size */
    BD_ERR_CUDA = 7,        /* a CUDA runtime call or launch failed */
    BD_ERR_TIMEOUT = 8,     /* device: a bounded wait inside a kernel ran out */
    BD_ERR_UNSUPPORTED = 9  /* the requested kernel path cannot run this shape */
} bd_status;

typedef enum { BD_F32 = 0, BD_BF16 = 1 } bd_dtype;

/* Kernel path for bitdelta_linear_ex (bitdelta_linear picks automatically). */
typedef enum {
    BD_PATH_AUTO = 0,
    BD_PATH_SIMT = 1,       /* CUDA-core kernel, any M */
    BD_PATH_DECODE_TC = 2,  /* tcgen05 decode kernel: base and sign products on tensor cores;
                               M <= 176 tokens.  With 2 to 8 K slices and M <= 128 the slices
                               of a 128-row tile launch as one thread-block cluster */
    BD_PATH_PREFILL_TC = 3, /* tcgen05 prefill kernel.  With at least 2048 tokens per present
                               variant (M / min(V, M) >= 2048, and at most 32 GiB of W_eff) every
                               present variant's W_eff (nearest bf16) is first written to the
                               workspace, one HBM pass per variant, and the GEMM loads it; with
                               fewer tokens bf16 W_eff tiles are built in shared memory */
    BD_PATH_DECODE_FOLD = 4, /* tcgen05 decode kernel with one sign accumulator shared by all
                               variants (a column per token), the scales applied in the epilogue:
                               M <= 128 tokens and at most 16 distinct variants */
    BD_PATH_DECODE_WEFF = 5 /* tcgen05 decode kernel for a single variant (V == 1): bf16 W_eff
                               tiles built in shared memory, the activations used as they are;
                               M <= 128 tokens, K % 64 == 0 */
} bd_path;

/* ------------------------------------------------------------------ */
/* Compression ("The mathematical foundation": the delta, the scale    */
/* alpha = (1/n)*||delta||_1 with n = N*K, and sign(delta) kept as one */
/* bit; "Infrastructure details": bits packed 8 per byte, alpha f32). */
/* ------------------------------------------------------------------ */

/* Bytes of device workspace bitdelta_compress needs for an N x K matrix on
 * the current device.  Returns 0 for invalid sizes. */
size_t bitdelta_compress_workspace(int64_t N, int64_t K);

/* Compress one fine-tuned matrix against its base.
 *   w_ft, w_base : device, [N, K] row-major, both of dtype in_dtype
 *                  (BD_F32 or BD_BF16); inputs are assumed finite (a NaN
 *                  gives bit 0 and a NaN alpha).
 *   N, K         : N >= 1, K >= 32, K % 32 == 0.
 *   alpha_out    : device, 1 float: the f32 nearest to the mean of
 *                  |W_ft - W_base| over all N*K entries (summed in fp32
 *                  partials of 32 terms and fp64 beyond; deterministic for a
 *                  given device and shape).
 *   bits_out     : device, N*K/32 u32 words in the packed layout above.
 *   workspace    : device, ws_bytes >= bitdelta_compress_workspace(N, K).
 * Returns BD_OK, or an argument error with nothing launched. */
bd_status bitdelta_compress(const void *w_ft, const void *w_base, bd_dtype in_dtype,
                            int64_t N, int64_t K, float *alpha_out, uint32_t *bits_out,
                            void *workspace, size_t ws_bytes, void *stream);

/* Per-output-row scale ("Infrastructure details": alpha stored as f32, one
 * per output dimension): alpha_out[n] = f32(mean_k |W_ft[n,k] - W_base[n,k]|),
 * bits as bitdelta_compress.  alpha_out: device, N floats.  Needs no
 * workspace; rows are independent. */
bd_status bitdelta_compress_rows(const void *w_ft, const void *w_base, bd_dtype in_dtype,
                                 int64_t N, int64_t K, float *alpha_out, uint32_t *bits_out,
                                 void *stream);

/* bitdelta_compress for callers that cannot allocate device memory (an
 * engine whose pool owns all device memory, a plugin that must not grow the
 * footprint, a path where an allocation would synchronise the device).  The
 * page has no counterpart: this is an interface convenience, not part of the
 * method.  Arguments and results are those of bitdelta_compress minus the
 * workspace; the scratch (one fp64 partial per block, at most 2048 blocks,
 * 16.6 KB) is a static device array inside the library that every GPU
 * loading the library keeps until the process exits.
 *   - Every call looks up that array's device address with the current
 *     device (no allocation).  The first call on a device, and the first
 *     after a reset of its context, loads the library's device code; make
 *     that call before any stream capture.
 *   - All calls share the array and it keeps the last call's contents; the
 *     finishing ticket is cleared on the stream before every launch.  Calls
 *     that overlap on the GPU race on the array: order them on one stream.
 *   - The launch uses at most 2048 blocks (one partial each); larger
 *     matrices are covered by the kernel's grid-stride loop, so any size that
 *     bitdelta_compress takes is accepted.
 * Calls no allocating routine. */
bd_status bitdelta_compress_noalloc(const void *w_ft, const void *w_base, bd_dtype in_dtype,
                                    int64_t N, int64_t K, float *alpha_out,
                                    uint32_t *bits_out, void *stream);

/* Materialised effective weights of one variant ("Serving architecture":
 * the conceptual listing rebuilds W_eff in the base dtype and hands it to a
 * standard linear; "Latency profile": reconstruction in prefill, then the
 * standard matmul).  The fused linear below never needs this; it exists so
 * that "reconstruct, then a library GEMM" can run beside the fused path.
 *   W_eff[n,k] = bf16(W_base[n,k] + a * s[n,k]), rounded to nearest (ties to
 *   even) from the exact sum; a = alpha[0] (per_row == 0) or alpha[n]
 *   (per_row != 0); s = +1 where the stored bit is 1, -1 where it is 0.
 *   w_base    : device, bf16 [N, K] row-major, 16-byte aligned.
 *   alpha     : device, float [1] or [N].
 *   bits      : device, [N, K/32] words as bitdelta_compress writes them.
 *   w_eff_out : device, bf16 [N, K], 16-byte aligned, not overlapping w_base.
 *   N >= 1, K >= 32, K % 32 == 0.
 * Returns BD_OK, or an argument error (overlap: BD_ERR_ALIGN) with nothing
 * launched. */
bd_status bitdelta_reconstruct(const void *w_base, const float *alpha, int32_t per_row,
                               const uint32_t *bits, int64_t N, int64_t K,
                               void *w_eff_out, void *stream);

/* ------------------------------------------------------------------ */
/* Multi-variant fused linear ("Serving architecture": W_eff =         */
/* W_base + alpha_v * sign(delta_v), reconstructed on the fly and fused */
/* with the matmul; the decode paths never write it to HBM, the prefill */
/* path may, see BD_PATH_PREFILL_TC).                                   */
/* ------------------------------------------------------------------ */

/* Bytes of device workspace bitdelta_linear needs for this shape.  Besides
 * the grouping and the staged activations of the tensor-core paths this
 * includes, when the prefill path would materialise W_eff (M / min(V, M) >=
 * 2048 tokens per present variant), min(V, M) * N * K * 2 bytes for the
 * materialised bf16 weights -- 1.9 GB for four variants of a 28672 x 8192
 * matrix. */
size_t bitdelta_linear_workspace(int64_t M, int64_t N, int64_t K, int32_t V);

/* y[t, n] = sum_k x[t,k] * (W_base[n,k] + alpha_{v(t)} * s_{v(t)}[n,k]),
 * s = +1 where the stored bit is 1 and -1 where it is 0, v(t) =
 * variant_ids[t]; a token with id -1 uses the base weights only.
 *   x           : device, bf16 [M, K].
 *   variant_ids : device, int32 [M], each in [-1, V).  A token whose id is
 *                 outside that range gets an all-zero row of y and sets
 *                 BD_ERR_VARIANT in the workspace status word.
 *   M, N, K     : M >= 0 (M == 0 is a no-op), N >= 1, K >= 32, K % 32 == 0.
 *   w_base      : device, bf16 [N, K].
 *   alphas      : device, float [V]: the per-matrix scale of each variant.
 *   bits        : HOST array of V device pointers, each to that variant's
 *                 packed [N, K/32] words.  Read during the call only.
 *   V           : 0 <= V <= BITDELTA_MAX_VARIANTS.
 *   y           : device, [M, N] of y_dtype (BD_F32 or BD_BF16), rows in the
 *                 original token order.  Accumulation is fp32 in every path.
 *   workspace   : device, ws_bytes >= bitdelta_linear_workspace(M, N, K, V).
 */
bd_status bitdelta_linear(const void *x, const int32_t *variant_ids,
                          int64_t M, int64_t N, int64_t K,
                          const void *w_base, const float *alphas,
                          const uint32_t *const *bits, int32_t V,
                          void *y, bd_dtype y_dtype,
                          void *workspace, size_t ws_bytes, void *stream);

/* Group the tokens of one batch by variant id ("Serving architecture": each
 * request names its variant; grouping lets one pass read each distinct
 * variant's bits once per weight tile): a stable counting sort of
 * variant_ids into the grouping area of `workspace`.  All linears of one
 * decode step see the same ids, so a caller may group once and then call
 * bitdelta_linear_grouped for every linear of the step.
 *   variant_ids : device, int32 [M]; ids outside [-1, V) set BD_ERR_VARIANT
 *                 in the status word and their output rows are zeroed.
 *   workspace   : device, at least bitdelta_linear_workspace(M, N, K, V)
 *                 bytes for the largest (N, K) it will serve; the grouping
 *                 area depends on M and V only. */
bd_status bitdelta_group(const int32_t *variant_ids, int64_t M, int32_t V,
                         void *workspace, size_t ws_bytes, void *stream);

/* The fused linear on a batch already grouped by bitdelta_group (same
 * workspace, same M and V, on the same stream).  Arguments as
 * bitdelta_linear, plus an explicit kernel path. */
bd_status bitdelta_linear_grouped(const void *x, int64_t M, int64_t N, int64_t K,
                                  const void *w_base, const float *alphas,
                                  const uint32_t *const *bits, int32_t V,
                                  void *y, bd_dtype y_dtype,
                                  void *workspace, size_t ws_bytes, void *stream,
                                  bd_path path);

/* bitdelta_linear with an explicit kernel path (for tests and measurement).
 * A path that cannot run the shape returns BD_ERR_UNSUPPORTED. */
bd_status bitdelta_linear_ex(const void *x, const int32_t *variant_ids,
                             int64_t M, int64_t N, int64_t K,
                             const void *w_base, const float *alphas,
                             const uint32_t *const *bits, int32_t V,
                             void *y, bd_dtype y_dtype,
                             void *workspace, size_t ws_bytes, void *stream,
                             bd_path path);

/* The fused linear with one scale per (variant, output row) ("Infrastructure
 * details": the scales are stored as f32, one per output dimension), the
 * form bitdelta_compress_rows produces:
 *   y[t, n] = sum_k x[t,k] * (W_base[n,k] + alpha_rows[v(t) * N + n] * s_{v(t)}[n,k]).
 *   alpha_rows : device, float [V, N] row-major (variant v's scales start at
 *                alpha_rows + v * N), 4-byte aligned.
 * Other arguments, layouts, ownership, errors and kernel paths as
 * bitdelta_linear_ex (every path takes per-row scales). */
bd_status bitdelta_linear_rows(const void *x, const int32_t *variant_ids,
                               int64_t M, int64_t N, int64_t K,
                               const void *w_base, const float *alpha_rows,
                               const uint32_t *const *bits, int32_t V,
                               void *y, bd_dtype y_dtype,
                               void *workspace, size_t ws_bytes, void *stream,
                               bd_path path);

/* ------------------------------------------------------------------ */
/* Status                                                               */
/* ------------------------------------------------------------------ */

/* Synchronise `stream`, read the status word at the start of `workspace`
 * (any workspace given to bitdelta_compress or bitdelta_linear), clear it,
 * and return the lowest-numbered error it holds (BD_OK if none). */
bd_status bitdelta_device_status(void *workspace, void *stream);

/* Health check of the bounded waits inside the tensor-core kernels (the page
 * has no counterpart; this is failure-detection plumbing).  One GPU thread
 * waits on a barrier for `poll_limit` polls (1 .. 2^24).  With arrive != 0 the
 * barrier completes first and nothing is reported; with arrive == 0 nothing
 * arrives, the wait runs out and BD_ERR_TIMEOUT is OR-ed into the status word
 * of `workspace` (any linear or compress workspace, >= 256 bytes), exactly as
 * a stalled pipeline inside a kernel would report it.  Read it with
 * bitdelta_device_status.  The device stays usable. */
bd_status bitdelta_check_bounded_wait(void *workspace, uint32_t poll_limit, int arrive,
                                      void *stream);

/* Kernels this library has enqueued since it was loaded, over all devices
 * and streams (launches that failed included).  Measurement plumbing; the
 * page has no counterpart.  Thread-safe; reading it costs no GPU work. */
uint64_t bitdelta_launch_count(void);

/* Static English text for a status code. */
const char *bitdelta_status_string(bd_status s);

/* BITDELTA_ABI_VERSION of the loaded library. */
int bitdelta_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BITDELTA_H */

/*
 * fckl.h -- C-ABI of the fused chunked KL distillation loss for NVIDIA B300 (sm_103a).
 *
 * The operation.  A student is distilled from a teacher whose output was cached
 * offline as its top-K (id, logit) pairs per token position (axbrief.com,
 * "Breaking the Bottleneck with Offline Caching and Chunked Loss";
 * getaibook.com, "Preparing Offline Top-K Logits").  The loss is the KL
 * divergence between teacher and student (getaibook.com, "Configuring Fused
 * Chunked KL Loss"), with the student's output projection (lm_head) folded
 * into it, so the [tokens x vocab] logit grid is never built, and the
 * sequence is processed one chunk at a time (calcaas.com, "What actually
 * changed?").  The pages print no formula; this library computes, for every
 * row t with the tempered student logits s_t = (H_t . W^T) / tau:
 *
 *   log p_tk = a_tk - logsumexp_k(a_t),   a_tk = topk_logits_tk / tau
 *   lse_t    = logsumexp_v(s_tv)
 *   loss_t   = sum_k p_tk (log p_tk - s_t,idx_tk + lse_t)       (forward KL)
 *   loss     = sum_{valid t} loss_t / N,     N = number of valid rows
 *   dz_tv    = g (exp(s_tv - lse_t) - sum_k p_tk [idx_tk = v]) / (tau N)
 *   dH = dz . W,   dW = dz^T . H
 *
 * with g = grad_loss (times *grad_scale when given); N = 0 gives loss 0 and
 * zero gradients.  Duplicate ids in a row add up termwise.  A cached logit of
 * -inf marks a pair the cache does not hold (a row with fewer than K pairs):
 * its p is 0 and it adds nothing to loss_t (the sum runs over p_tk > 0, as
 * 0 log 0 = 0), which is the same as leaving it out.  Every valid row needs at
 * least one finite logit.  Ignored rows (valid[t] == 0) add nothing to the
 * loss, their dH rows are exactly 0 and they add nothing to dW whatever their
 * topk_logits hold (NaN and +-inf included); their ids must still lie in
 * [0, V).  H and W must be finite.
 *
 * Conventions shared by every call:
 *  - All tensors are row-major and contiguous, on the current CUDA device.
 *    H[T, d] and W[V, d] hold `dtype` elements; dH[T, d] is written in the
 *    same dtype; dW[V, d] is float32.  topk_idx[T, K] is int32 in [0, V);
 *    topk_logits[T, K] float32; valid[T] uint8 (nonzero = the row counts);
 *    lse[T] and row_loss[T] float32.
 *  - The caller owns every buffer.  The library never allocates device
 *    memory: scratch space is the caller's workspace `ws` of at least
 *    fckl_workspace_size(...) bytes, 256-byte aligned.  No state is kept
 *    between calls except the optional launch counters and profiling events
 *    of the instrumentation calls at the end of this header.
 *  - Every compute call is asynchronous and stream-ordered on `stream` (a
 *    cudaStream_t; NULL = the legacy default stream).  Calls that share a
 *    workspace must be ordered on the GPU.
 *  - Argument errors are returned before anything is launched.  Errors the
 *    GPU detects (an id outside [0, V), a wait that timed out) are recorded in
 *    a status word inside the workspace; read them with fckl_get_error after
 *    the work, no kernel ever traps.  fckl_forward clears that word first.
 *  - bf16 work runs on tcgen05 tensor cores (bf16 inputs, fp32 accumulation)
 *    and needs d % 8 == 0 and 16-byte aligned H, W, dH; float32 work runs on
 *    fp32 CUDA cores.
 */
#ifndef FCKL_H_
#define FCKL_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FCKL_API __attribute__((visibility("default")))
#else
#define FCKL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FCKL_OK = 0,
  FCKL_ERR_INVALID_ARG = 1, /* a null pointer, a size or tau out of range */
  FCKL_ERR_UNSUPPORTED = 2, /* valid arguments this build cannot run (alignment, K limit, device) */
  FCKL_ERR_WORKSPACE = 3,   /* ws is null, too small or not 256-byte aligned */
  FCKL_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch, attribute, memset) */
  FCKL_ERR_BAD_INDEX = 5,   /* a teacher id outside [0, V) (reported by fckl_get_error) */
  FCKL_ERR_TIMEOUT = 6      /* a bounded on-device wait gave up (reported by fckl_get_error) */
} fckl_status;

typedef enum { FCKL_F32 = 0, FCKL_BF16 = 1 } fckl_dtype;

/* Largest K (teacher ids per row) the kernels accept. */
#define FCKL_MAX_K 1024

/* Bytes of workspace fckl_forward and fckl_backward need for these sizes (the
 * same for both).  It grows with the chunk (per-chunk scratch of
 * O(chunk * vocab tile)), never with T * V; 0 for invalid sizes. */
FCKL_API size_t fckl_workspace_size(int64_t T, int64_t d, int64_t V, int32_t K, int64_t chunk,
                           fckl_dtype dtype);

/* Forward: the mean loss and the per-row student logsumexp.
 * Processes the T rows `chunk` rows at a time; for each chunk the logit tiles
 * H_chunk . W^T are formed tile by tile and reduced on chip to a running
 * max / sum per row and to the student logits at the teacher's ids, so the
 * result does not depend on `chunk`.
 *   loss     device float32 scalar, written (0 when no row is valid)
 *   lse      device float32 [T], written for every row, ignored rows included
 *            (logsumexp of s_t = H_t . W^T / tau; fckl_backward takes it back)
 *   row_loss device float32 [T] or NULL: loss_t for valid rows, 0 for ignored
 * Returns FCKL_OK once the work is queued on `stream`. */
FCKL_API fckl_status fckl_forward(const void* H, const void* W, const int32_t* topk_idx,
                         const float* topk_logits, const uint8_t* valid, int64_t T, int64_t d,
                         int64_t V, int32_t K, float tau, int64_t chunk, fckl_dtype dtype,
                         float* loss, float* lse, float* row_loss, void* ws, size_t ws_bytes,
                         void* stream);

/* Backward: dH and dW of g * loss, recomputing the logit tiles chunk by chunk
 * (the extra projection work in the backward pass that chunking costs,
 * axbrief.com, "Breaking the Bottleneck with Offline Caching and Chunked Loss").
 * A chunk is worked through in row blocks of at most 4096 rows (all of it when the chunk
 * is smaller), each block over every vocab stripe; the chunk bounds the workspace.
 *   lse        device float32 [T] from fckl_forward with the same inputs
 *   grad_loss  host scalar g (dL/dloss)
 *   grad_scale device float32 scalar or NULL; when given, g is multiplied by it
 *   dH         device [T, d] in `dtype`, overwritten; rows of ignored tokens are 0
 *   dW         device float32 [V, d], overwritten
 * Reproducibility: loss, lse and dW are bit for bit the same from run to run.  On the bf16
 * path dH is accumulated in float32 by one reduce-add per vocab stripe, and tiles of
 * consecutive stripes run at the same time, so the order of those adds (and the last bits
 * of dH) can change from run to run.
 * Returns FCKL_OK once the work is queued on `stream`. */
FCKL_API fckl_status fckl_backward(const void* H, const void* W, const int32_t* topk_idx,
                          const float* topk_logits, const uint8_t* valid, int64_t T, int64_t d,
                          int64_t V, int32_t K, float tau, int64_t chunk, fckl_dtype dtype,
                          const float* lse, float grad_loss, const float* grad_scale, void* dH,
                          float* dW, void* ws, size_t ws_bytes, void* stream);

/* Teacher top-K extraction, the offline step that builds the cache the loss reads: the
 * teacher is run once and only its K largest logits per token position are kept, with
 * their ids (getaibook.com, "Preparing Offline Top-K Logits"; axbrief.com, "Breaking the
 * Bottleneck with Offline Caching and Chunked Loss").  For every row t of logits[T, V]
 * (`dtype` elements, row-major, contiguous) writes the K entries that come first in the
 * order value descending, then id ascending:
 *   topk_idx    device int32 [T, K]: their ids, in that order
 *   topk_logits device float32 [T, K]: their values widened to float32 (exact)
 * so the output is unique even where values tie, and is the topk_idx / topk_logits input
 * of fckl_forward as is.  Values are ordered by their bit patterns read as sign-magnitude
 * numbers: numeric order for all non-NaN values, -0 just below +0, NaNs with the sign bit
 * clear above +inf and with it set below -inf.  Needs 1 <= K <= min(V, FCKL_MAX_K) and
 * V < 2^31 (FCKL_ERR_INVALID_ARG), logits aligned to its element size and the outputs to
 * 4 bytes (FCKL_ERR_UNSUPPORTED).  Allocates nothing and keeps no state; asynchronous on
 * `stream`; returns FCKL_OK once the work is queued. */
FCKL_API fckl_status fckl_topk_extract(const void* logits, int64_t T, int64_t V, int32_t K, fckl_dtype dtype,
                                       int32_t* topk_idx, float* topk_logits, void* stream);

/* ---- token-sharded data parallelism ---------------------------------------------------
 * The pages place the method in distillation runs that would otherwise be spread over many
 * GPUs and nodes (getaibook.com, "Hardware and Performance Tradeoffs"; axbrief.com,
 * "Quantifying the Efficiency Gain: 15.6x VRAM Reduction").  The loss shards over tokens:
 * each rank runs fckl_forward / fckl_backward on its own rows (H, topk_idx, topk_logits,
 * valid) with the whole W.  Three things cross ranks: the loss sum and N, which the mean
 * and the gradient scale g / (tau N) need over all ranks, and dW, which sums over ranks;
 * dH stays with its rank.  These two calls hand the first two to the caller's collective
 * (a sum over ranks, e.g. an all-reduce) and back; dW is summed by the caller as is.
 *
 * Writes partials (device double[2], 8-byte aligned) = { sum of loss_t over the valid rows,
 * N } of the last fckl_forward on workspace `ws`, stream-ordered after it. */
FCKL_API fckl_status fckl_loss_partials(const void* ws, size_t ws_bytes, double* partials, void* stream);

/* From total (device double[2]: the partials summed over ranks) and this rank's own partials
 * `local`, writes
 *   loss       device float32 scalar: total[0] / total[1], the mean over all ranks' valid
 *              rows (0 when total[1] == 0)
 *   grad_scale device float32 scalar: local[1] / total[1] (0 when total[1] == 0); passed as
 *              fckl_backward's grad_scale on this rank, it makes the gradient scale
 *              g / (tau N_total), so that the ranks' dW add up to the whole batch's.
 * Asynchronous on `stream`. */
FCKL_API fckl_status fckl_loss_finish(const double* total, const double* local, float* loss, float* grad_scale,
                                      void* stream);

/* dst[i] = src[i] rounded to bfloat16 (to nearest, ties to even), for i < n: for a caller
 * holding dW in float32 whose weights are bf16 (an autograd gradient takes the weights'
 * dtype).  The pages have no counterpart: it is the cast at the end of the user's backward.
 * Needs n % 4 == 0, src 16-byte and dst 8-byte aligned (FCKL_ERR_UNSUPPORTED), n >= 0 and
 * non-null pointers when n > 0 (FCKL_ERR_INVALID_ARG).  Asynchronous on `stream`. */
FCKL_API fckl_status fckl_cast_f32_to_bf16(const float* src, void* dst, int64_t n, void* stream);

/* Waits for `stream`, then returns and clears the status word the GPU wrote in
 * the workspace (FCKL_OK, FCKL_ERR_BAD_INDEX or FCKL_ERR_TIMEOUT), or
 * FCKL_ERR_CUDA when the wait or the copy itself failed. */
FCKL_API fckl_status fckl_get_error(void* ws, void* stream);

/* A static description of a status code. */
FCKL_API const char* fckl_status_string(fckl_status status);

/* ---- instrumentation (host-side counters; off unless enabled) ---------------------------
 * Kernel classes, in the order the path runs them. */
typedef enum {
  FCKL_K_PREP = 0,     /* teacher softmax + id sort, per chunk */
  FCKL_K_FWD_TILES,    /* logit tiles + online max/sum + gather (forward) */
  FCKL_K_COMBINE,      /* per-row lse and loss_t from the tile partials */
  FCKL_K_REDUCE,       /* fixed-order mean over rows; N and the gradient scale */
  FCKL_K_BWD_TILES,    /* backward: recomputed logit tiles -> gradient tile G; on the bf16
                          path the same launch also runs dW (+)= G^T . H_chunk and
                          dH_chunk += G . W for every vocab stripe of the chunk */
  FCKL_K_GRAD_GEMM,    /* dW / dH contractions launched on their own (fp32 path) */
  FCKL_K_OTHER,        /* memsets and casts */
  FCKL_K_TOPK,         /* teacher top-K extraction (fckl_topk_extract) */
  FCKL_K_NUM_CLASSES
} fckl_kernel_class;

/* Number of kernels this library has launched since load (all classes). */
FCKL_API int64_t fckl_launch_count(void);

/* When on, every launch is bracketed by CUDA events on its stream so that
 * fckl_profile_read can report per-class device time.  Off by default. */
FCKL_API void fckl_profile_enable(int on);

/* Synchronizes the recorded events and returns, for one class, the number of
 * launches and their summed device time (ms) since the last reset; resets
 * when `reset` is nonzero.  Returns FCKL_ERR_INVALID_ARG for a bad class. */
FCKL_API fckl_status fckl_profile_read(int32_t kernel_class, int64_t* launches, double* total_ms, int reset);

/* Test hook for the failure path: launches one thread that waits, with the kernels' own
 * bounded wait, on a barrier nothing arrives on.  After FCKL_WAIT_NS (2 s) the wait gives up
 * and records FCKL_ERR_TIMEOUT in the workspace's status word, which fckl_get_error then
 * returns; nothing faults or hangs.  ws: a workspace of at least 256 bytes. */
FCKL_API fckl_status fckl_debug_wait_timeout(void* ws, size_t ws_bytes, void* stream);

/* Test hook for the tcgen05 GEMM engine: D[M, N] (float32, row-major, ldd = N)
 * = A . B with bf16 operands on the same tensor-core path the loss uses.
 * a_mn == 0: A is [M, K] (K contiguous); a_mn == 1: A is stored [K, M].
 * b_mn == 0: B is stored [N, K] (so D = A . B^T); b_mn == 1: B is stored [K, N].
 * cta_pair != 0 runs 256-row tiles on CTA pairs (cta_group::2), the engine the loss uses;
 * 0 runs 128-row tiles on single CTAs.  The pair engine takes only b_mn == 0
 * (FCKL_ERR_UNSUPPORTED otherwise).
 * M, N, K >= 1; M or N contiguous extents need multiples of 8 elements. */
FCKL_API fckl_status fckl_debug_gemm_bf16(const void* A, const void* B, float* D, int64_t M, int64_t N,
                                 int64_t K, int32_t a_mn, int32_t b_mn, int32_t cta_pair, void* stream);

/* ---- forward without a workspace --------------------------------------------------------
 * The pages describe no such call: it has no counterpart in the method and exists only for
 * callers of this library that cannot allocate device memory.  Such callers include code
 * running while a CUDA stream is being captured into a graph (cudaMalloc is refused during
 * capture), runtimes that reserve all device memory up front for their own pool and hand
 * library code nothing but the buffers they own (a foreign cudaMalloc then fails), and
 * latency-critical loops that cannot risk the device-wide synchronization cudaMalloc and
 * cudaFree may cause.
 *
 * Size of the scratch array fckl_forward_noalloc keeps in the library's own device memory.
 * Every GPU that loads the library holds this much until the process exits. */
#define FCKL_NOALLOC_SCRATCH_BYTES (8u << 20)

/* fckl_forward with the same arguments and results, except that it takes no workspace and
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine).  Its scratch
 * is a fixed FCKL_NOALLOC_SCRATCH_BYTES array in the library's device memory, so it needs
 * the per-row loss output and an optional status output from the caller:
 *   row_loss  device float32 [T], required when T > 0 (loss_t, 0 for ignored rows)
 *   status    device int32 scalar or NULL; receives the status word of this call
 *             (FCKL_OK, FCKL_ERR_BAD_INDEX or FCKL_ERR_TIMEOUT) once the work is done
 * Rows are processed in chunks of at most `chunk` rows, smaller when a chunk's scratch
 * (16*K + 8*ceil(V/256) bytes per row) would not fit; the results do not depend on the
 * chunk size.  Returns FCKL_ERR_WORKSPACE when a single row's scratch exceeds
 * FCKL_NOALLOC_SCRATCH_BYTES, before anything is launched.
 * Every call looks up the array's device address on the current device; the first call on
 * a device may also load the library's GPU code, so make that first call before any stream
 * capture.  All calls share
 * the one array, which keeps the last call's contents: the call clears what must start at
 * zero itself, but calls that overlap on the GPU (other streams or host threads on the
 * same device) race on it and must be serialized by the caller. */
FCKL_API fckl_status fckl_forward_noalloc(const void* H, const void* W, const int32_t* topk_idx,
                                          const float* topk_logits, const uint8_t* valid, int64_t T,
                                          int64_t d, int64_t V, int32_t K, float tau, int64_t chunk,
                                          fckl_dtype dtype, float* loss, float* lse, float* row_loss,
                                          int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FCKL_H_ */

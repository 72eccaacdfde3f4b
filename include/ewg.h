/*
 * ewg.h -- C ABI of the GB300 sparse embedding weight-gradient library.
 *
 * The operation (Megatron Core API docs, core.fusions.fused_embedding_wgrad,
 * entry accumulate_embedding_wgrad, and the module docstring):
 *
 *     main_grad += embedding_dense_backward(grad, ids)
 *
 * touching only the rows of the ids that occur.  The values are those of PyTorch's
 * sort-based embedding backward followed by main_grad.add_ (module docstring,
 * both bullets): the (token, position) pairs are sorted; each token's gradient rows
 * are summed in position order into fp32 partial sums of at most EWG_NROWS rows,
 * chunked from the token's first row; the partial sums are added in order starting
 * from 0; the total is rounded once to the gradient dtype; that value is added to
 * the main_grad row in fp32 and rounded to main_grad's dtype.  Rows of ids that do
 * not occur are neither read nor written (module docstring, last sentence).
 * Every rounding is IEEE round-to-nearest-even; results are deterministic and
 * independent of the launch configuration.
 *
 * Conventions for every entry point below:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or keeps them.  All tensors must live on the current
 *     CUDA device.
 *   - "stream" is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Work is enqueued on it and the call returns without waiting for it.
 *   - Errors a host check can find are returned BEFORE anything is enqueued, so
 *     main_grad is untouched.  Errors found on the device (an id outside
 *     [0, num_embeddings)) make every kernel of the call skip all writes to
 *     main_grad; ewg_read_status() reports them.
 *   - No C++ exception crosses this boundary.  Entry points are thread-safe; two
 *     calls that share a workspace or a main_grad must be ordered by the caller
 *     (same stream, or events).
 */
#ifndef EWG_H_
#define EWG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Fewest tokens accepted: PyTorch's embedding backward takes its sort-based path,
 * whose arithmetic this library reproduces, only above 3072 tokens (module
 * docstring, first bullet; MIN_TOKENS = 3073 on the same page). */
#define EWG_MIN_TOKENS 3073
/* Most tokens accepted.  The page's own limit is 8192 (MAX_TOKENS), set by its
 * single-program sort; this library sorts across many CTAs and keeps 32-bit slot
 * indices, so it accepts up to 2^28 tokens. */
#define EWG_MAX_TOKENS (1 << 28)
/* Partial-sum chunk length (NROWS on the page, NROWS_PER_THREAD in PyTorch). */
#define EWG_NROWS 10
/* Largest hidden size accepted. */
#define EWG_MAX_HIDDEN (1 << 24)

/* Element types (ewg_dtype). */
#define EWG_INT32 0
#define EWG_INT64 1
#define EWG_BF16 2
#define EWG_FP32 3

/* Status codes (ewg_status). */
#define EWG_OK 0
#define EWG_ERR_UNSUPPORTED 1     /* tensors outside what ewg_can_accumulate accepts */
#define EWG_ERR_INVALID 2         /* bad argument: NULL, size, workspace too small, plan mismatch */
#define EWG_ERR_CUDA 3            /* a CUDA runtime call or kernel launch failed */
#define EWG_ERR_ID_OUT_OF_RANGE 4 /* device-detected: an id outside [0, num_embeddings) */
#define EWG_ERR_TIMEOUT 5         /* device-detected: a bounded wait in a kernel gave up;
                                     touched main_grad rows are then unspecified */
#define EWG_ERR_BOUNDS 6          /* device-detected, bounds-checking build (libewg_debug.so)
                                     only: an index a kernel derived from the plan was out of
                                     range; the access was replaced by a safe one, so
                                     main_grad's touched rows are then unspecified */

/*
 * Whether ewg_accumulate supports these tensors (can_accumulate_embedding_wgrad on
 * the page).  Returns 1 or 0 and never enqueues work.
 *
 *   ids        [num_tokens] contiguous, ids_dtype EWG_INT32 or EWG_INT64.  A
 *              multi-dimensional ids tensor is passed flattened in row-major order;
 *              token position p is its flat index.
 *   grad       [num_tokens][hidden], grad_dtype EWG_BF16 or EWG_FP32, unit inner
 *              stride, grad_row_stride elements between rows (>= hidden).
 *   main_grad  [num_embeddings][hidden], EWG_BF16 or EWG_FP32, unit inner stride,
 *              main_grad_row_stride elements between rows (>= hidden).
 *
 * Conditions: EWG_MIN_TOKENS <= num_tokens <= EWG_MAX_TOKENS;
 * 1 <= num_embeddings < 2^31; 8 <= hidden <= EWG_MAX_HIDDEN and hidden % 8 == 0;
 * grad, main_grad and their row strides 16-byte aligned; ids aligned to its element;
 * all three pointers are device (or managed) memory of the current device;
 * main_grad does not overlap grad or ids.  The page's further conditions (Triton
 * present, ids and positions packing into 31 bits, at most 8192 tokens) belong to
 * its own implementation and are not imposed here.
 */
int ewg_can_accumulate(const void* ids, int ids_dtype, int64_t num_tokens,
                       const void* grad, int grad_dtype, int64_t grad_row_stride,
                       const void* main_grad, int main_grad_dtype,
                       int64_t num_embeddings, int64_t hidden,
                       int64_t main_grad_row_stride);

/*
 * Bytes of device workspace that ewg_accumulate / ewg_plan / ewg_apply need for
 * num_tokens tokens of width hidden (an upper bound over every id pattern).  The page
 * has no counterpart: its function allocates its own scratch, while this library leaves
 * every allocation to the caller.  The workspace needs no initialisation and holds no
 * state the caller must keep between calls, except that ewg_apply reads the plan that
 * ewg_plan left in it and ewg_read_status reads the status of the last call.  Returns 0
 * for sizes outside the supported range.
 */
size_t ewg_workspace_bytes(int64_t num_tokens, int64_t hidden);

/*
 * main_grad += embedding_dense_backward(grad, ids), touching only the rows of ids
 * (accumulate_embedding_wgrad on the page).  Arguments as for ewg_can_accumulate,
 * plus a device workspace of at least ewg_workspace_bytes(num_tokens, hidden)
 * bytes, 256-byte aligned, and the stream.  Equivalent to ewg_plan followed by
 * ewg_apply on the same stream.
 *
 * Returns EWG_OK once the work is enqueued, EWG_ERR_UNSUPPORTED /
 * EWG_ERR_INVALID (nothing enqueued, main_grad untouched) or EWG_ERR_CUDA.
 * Out-of-range ids are found on the device: main_grad is then left untouched and
 * ewg_read_status returns EWG_ERR_ID_OUT_OF_RANGE.
 */
int ewg_accumulate(const void* ids, int ids_dtype, int64_t num_tokens,
                   const void* grad, int grad_dtype, int64_t grad_row_stride,
                   void* main_grad, int main_grad_dtype,
                   int64_t num_embeddings, int64_t hidden, int64_t main_grad_row_stride,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * The first half of ewg_accumulate (the page's _sort_tokens_kernel): validates the
 * ids on the device, sorts the (token, position) pairs, finds every token's run of
 * sorted slots and lists its chunks of at most EWG_NROWS rows, writing this plan
 * into the workspace.  Reads only ids; writes only the workspace.
 */
int ewg_plan(const void* ids, int ids_dtype, int64_t num_tokens, int64_t num_embeddings,
             int64_t hidden, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The second half of ewg_accumulate (the page's _partial_sums_kernel and
 * _long_run_sums_kernel): sums the chunks of the plan in the workspace and adds
 * each token's row into main_grad.  num_tokens, num_embeddings
 * and hidden must be those given to the ewg_plan that filled the workspace (the
 * kernel checks them against the plan and writes nothing on a mismatch, reporting
 * EWG_ERR_INVALID through ewg_read_status).  Must be ordered after that ewg_plan.
 */
int ewg_apply(const void* grad, int grad_dtype, int64_t grad_row_stride,
              void* main_grad, int main_grad_dtype, int64_t num_tokens,
              int64_t num_embeddings, int64_t hidden, int64_t main_grad_row_stride,
              void* workspace, size_t workspace_bytes, void* stream);

/*
 * Vocabulary-sharded ewg_accumulate: main_grad holds only the rows
 * [row_begin, row_begin + shard_rows) of the [num_embeddings, hidden] table (its row 0 is
 * table row row_begin), and the call updates exactly the rows of that range that
 * ewg_accumulate would update, with the same bits.  Ids in [0, num_embeddings) outside
 * the range are skipped; ids outside [0, num_embeddings) are errors as in
 * ewg_accumulate.
 *
 * The page has no entry point of its own for this.  It follows from the module
 * docstring of core.fusions.fused_embedding_wgrad: a row's result depends only on that
 * token's own rows, in position order, and rows of absent tokens are not touched, so
 * the rows of a range are computed the same way whatever happens to the other rows.
 * One GPU per range of rows then needs no exchange.
 *
 * ids, grad: as in ewg_accumulate (all num_tokens tokens; the support condition on
 * num_tokens is that of the whole call).  main_grad: shard_rows rows of hidden
 * elements, row stride main_grad_row_stride.  Requires 0 <= row_begin,
 * 1 <= shard_rows and row_begin + shard_rows <= num_embeddings (else
 * EWG_ERR_UNSUPPORTED before anything is enqueued).  Workspace, stream and errors:
 * as ewg_accumulate.
 */
int ewg_accumulate_shard(const void* ids, int ids_dtype, int64_t num_tokens,
                         const void* grad, int grad_dtype, int64_t grad_row_stride,
                         void* main_grad, int main_grad_dtype, int64_t num_embeddings,
                         int64_t row_begin, int64_t shard_rows, int64_t hidden,
                         int64_t main_grad_row_stride, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * The first half of ewg_accumulate_shard: ewg_plan keeping only the ids in
 * [row_begin, row_begin + shard_rows), renumbered from 0.  The ewg_apply that follows
 * takes num_embeddings = shard_rows and the shard's main_grad.
 */
int ewg_plan_shard(const void* ids, int ids_dtype, int64_t num_tokens,
                   int64_t num_embeddings, int64_t row_begin, int64_t shard_rows,
                   int64_t hidden, void* workspace, size_t workspace_bytes, void* stream);

/*
 * ewg_accumulate with ids and grad in pinned host memory (the page's function takes
 * device tensors; this is the same call for a caller whose inputs start on the host).
 *
 * ids_host: num_tokens ids (EWG_INT32 or EWG_INT64), contiguous; grad_host:
 * [num_tokens, hidden] (EWG_BF16 or EWG_FP32), contiguous (row stride = hidden).  Both
 * must be page-locked host memory (cudaHostAlloc / cudaHostRegister / a pinned torch
 * tensor), else EWG_ERR_UNSUPPORTED.  main_grad: a device matrix as in ewg_accumulate.
 * workspace: device memory of at least ewg_host_workspace_bytes(...) bytes; it receives
 * the copies of ids and grad next to the ordinary workspace.
 *
 * Stream-ordered on `stream`: the ids are copied and planned on `stream` while the grad
 * copy runs on a library-owned stream of the device (made on the first call, after the
 * work already queued on `stream`); the apply waits for both.  Calls on one device from
 * several host threads are serialised by the library while they enqueue.  Errors and
 * the device status: as ewg_accumulate (ewg_read_status on the same workspace).
 *
 * The copies read ids_host and grad_host after the call has returned: both buffers must
 * stay allocated and unchanged until `stream` has passed this call (synchronize it, or
 * wait on an event recorded on it after the call).
 *
 * The library keeps ONE copy stream per device for every caller stream, so the grad
 * copy of a call waits for the grad copies of earlier host-input calls on the same
 * device, whatever stream those were made on.
 */
size_t ewg_host_workspace_bytes(int64_t num_tokens, int64_t hidden, int ids_dtype,
                                int grad_dtype);
int ewg_accumulate_host(const void* ids_host, int ids_dtype, int64_t num_tokens,
                        const void* grad_host, int grad_dtype, void* main_grad,
                        int main_grad_dtype, int64_t num_embeddings, int64_t hidden,
                        int64_t main_grad_row_stride, void* workspace, size_t workspace_bytes,
                        void* stream);

/* Size of the library-owned scratch used by ewg_accumulate_static (64 MiB). */
#define EWG_STATIC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * ewg_accumulate without a caller workspace and without any allocation.  The page
 * (Megatron Core API docs, core.fusions.fused_embedding_wgrad) has no counterpart: this
 * is an addition for callers that cannot allocate.
 *
 * For callers that cannot allocate device memory when the gradient is accumulated:
 * code running under a fixed-pool or custom allocator that must not grow, and runtimes
 * that forbid cudaMalloc after start-up.  The library keeps a file-scope __device__ array of
 * EWG_STATIC_SCRATCH_BYTES as the workspace; every device that loads the library
 * holds it until the process exits.  Arguments and results are those of
 * ewg_accumulate, without the workspace.
 *
 * - Sizes whose ewg_workspace_bytes(num_tokens, hidden) exceeds
 *   EWG_STATIC_SCRATCH_BYTES are rejected with EWG_ERR_UNSUPPORTED (and
 *   ewg_last_error says so) before anything is enqueued.  64 MiB covers up to 8192
 *   tokens for hidden sizes up to about 10000.
 * - The call makes no cudaMalloc, cudaFree or other allocating call.  The first call on
 *   a device looks up the array's device address with cudaGetSymbolAddress; make that
 *   first call outside any stream capture.  Under CUDA's lazy module loading (the
 *   default) the array is reserved only then, when that lookup loads the module that
 *   holds it (with CUDA_MODULE_LOADING=EAGER, when the library is loaded): make the
 *   first call at start-up, while the device still has room for it.
 * - Every call on a device uses the same array, which keeps the last call's contents
 *   (nothing in it needs clearing between calls).  Calls that may overlap on the GPU
 *   (different streams without ordering) race on it and must not be made.
 * - If scratch_out is not NULL it receives the array's device address, which can be
 *   passed to ewg_read_status to read the device status of the call.
 */
int ewg_accumulate_static(const void* ids, int ids_dtype, int64_t num_tokens,
                          const void* grad, int grad_dtype, int64_t grad_row_stride,
                          void* main_grad, int main_grad_dtype,
                          int64_t num_embeddings, int64_t hidden,
                          int64_t main_grad_row_stride, void* stream, void** scratch_out);

/*
 * Waits for `stream`, then copies the device status of the last ewg_plan /
 * ewg_apply / ewg_accumulate that used this workspace into *status (EWG_OK,
 * EWG_ERR_ID_OUT_OF_RANGE, EWG_ERR_INVALID or EWG_ERR_TIMEOUT).  Returns EWG_OK or
 * EWG_ERR_CUDA.  The page has no counterpart: there an out-of-range id stops the
 * process with a device assertion, while here it is reported through this call (the
 * device-status query of the library's boundary).
 */
int ewg_read_status(const void* workspace, void* stream, int* status);

/* Human-readable name of a status code (static storage). */
const char* ewg_status_string(int status);

/* Detail of the last error returned on the calling thread (static storage, "" if none). */
const char* ewg_last_error(void);

/* Library ABI version. */
int ewg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EWG_H_ */

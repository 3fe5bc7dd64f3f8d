/*
 * fckl.h - C ABI of the fused, chunked top-K KL distillation loss on one GB300 (sm_103a).
 *
 * The operation ("Hugging Face：让知识蒸馏廉价到可大规模运行", paragraphs "离线蒸馏" and
 * "Fused, chunked KL loss"; "Chunkovaná KL strata umožnila destilovať LLM s 32-tisícovým
 * kontextom na jednom H200", sections "Dva odlišné zdroje úspory" and "Čo dopĺňajú
 * podrobnejšie experimenty"):
 *
 *   z_n    = W h_n                     student logits of position n, never stored whole
 *   lse_n  = log sum_v exp(z_nv)
 *   p_nk   = exp(logp_nk),  S_n = sum_k p_nk   (teacher top-K cache, not renormalised)
 *   loss   = sum_n sum_k p_nk (logp_nk - (z_{n,idx_nk} - lse_n))        (0 log 0 = 0)
 *   G_n    = S_n softmax(z_n) - p_sparse_n,   dH = G W,   dW = G^T H
 *
 * The sequence is walked one chunk of positions at a time: the forward pass projects
 * a chunk, folds it into the running loss and drops it; the backward pass recomputes
 * the chunk's logits to form G (the one-call path instead keeps, in the gradient slab itself,
 * what its backward needs of the chunk's logits, see fckl_forward_backward). Only one chunk x V
 * slab is ever held (two with the workspace of fckl_overlap_workspace_bytes).
 *
 * Conventions for every call below
 *  - All arrays are dense and row-major. "device" pointers are CUDA device memory of the
 *    current device; the caller owns every buffer, including the workspace. The library
 *    allocates no device memory at run time (the one exception is the fixed scratch array
 *    of fckl_forward_static, reserved when the library is loaded) and keeps only host-side
 *    caches (device properties, one-time kernel set-up) and, for fckl_forward_backward with
 *    the overlap workspace, one non-blocking CUDA stream and two events per host thread and
 *    device, created on first use and kept.
 *  - H is [N, d] and W is [V, d], both of type `dtype` (FCKL_BF16 or FCKL_F32). With FCKL_F32
 *    the logits products (the forward projection, the backward's recompute, both passes of
 *    the top-K builder) run on the tensor cores as tf32 with fp32 accumulation, on copies of
 *    W and of each chunk of H rounded to tf32 (10 explicit mantissa bits, to nearest, ties
 *    away from zero) in the workspace. G is rounded to bf16 as for bf16 inputs, and the dH
 *    and dW products read bf16 copies of W and of each chunk of H (round to nearest even).
 *    FCKL_BF16 inputs run every product in bf16 with fp32 accumulation.
 *  - idx is int32 [N, K]: teacher token ids, any order, each in [0, V). logp is fp32 [N, K]:
 *    the teacher's log-probabilities for those ids; -inf marks an empty slot. A repeated
 *    id within a row contributes once per slot.
 *  - weight is fp32 [N] or NULL (all ones): position n contributes weight[n] * loss_n to the
 *    loss and weight[n] * G_n to the gradients; 0 drops a padded position (sequence packing
 *    is among the ablations of "Hugging Face：让知识蒸馏廉价到可大规模运行", section "得到的
 *    student"). lse is not weighted.
 *  - `stream` is a cudaStream_t (may be NULL for the legacy default stream). Every call is
 *    asynchronous on it; inputs must stay alive and unmodified until the work completes.
 *  - Limits: 1 <= N <= 2^40, 1 <= K <= min(V, 1024), V <= 2^30, d % 8 == 0 (16-byte rows
 *    for the tensor memory accelerator) and d <= 2^20, 1 <= min(chunk, N) <= 2^24; H, W, dH
 *    and dW 16-byte aligned; ws 256-byte aligned.
 *  - Return value: FCKL_OK, or an fckl_status naming the first problem found. Argument
 *    errors launch nothing. Errors found on the device (a teacher id outside [0, V), a
 *    pipeline wait that ran out) cannot be returned by an asynchronous call: they are
 *    ORed into a status word in the workspace and read back by fckl_check().
 *    Results of a call whose status word is not clear are unspecified. No device code
 *    traps; every wait on the device is bounded in time.
 */
#ifndef FCKL_H
#define FCKL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FCKL_OK = 0,
    FCKL_ERR_ARG = 1,         /* bad size, null or misaligned pointer */
    FCKL_ERR_INDEX = 2,       /* a teacher id outside [0, V) (device-detected) */
    FCKL_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed; see fckl_last_error() */
    FCKL_ERR_TIMEOUT = 4,     /* a bounded device wait ran out (device-detected) */
    FCKL_ERR_WORKSPACE = 5,   /* ws_bytes below fckl_workspace_bytes() */
    FCKL_ERR_UNSUPPORTED = 6, /* shape outside the limits above, or not an sm_103 device */
    FCKL_ERR_CAPACITY = 7     /* teacher top-K: a position had more candidates than the buffer
                                 holds (device-detected; that position's output is not exact) */
} fckl_status;

typedef enum { FCKL_BF16 = 0, FCKL_F32 = 1 } fckl_dtype;

/* Bytes of device workspace that fckl_forward, fckl_backward and fckl_forward_backward need
 * for this shape ("Hugging Face：让知识蒸馏廉价到可大规模运行", paragraph "Fused, chunked KL
 * loss": only one chunk of positions is ever held, so memory never exceeds one chunk's size;
 * section "扩展到长上下文": peak memory grows linearly with the sequence length).
 * The size grows with chunk * V (the gradient slab) and with N only through 4 bytes per
 * position; for FCKL_F32 it also holds the tf32 and bf16 copies of W (6 * V * d bytes) and of
 * one chunk of H. 0 if the shape is outside the limits (including min(chunk, N) above 2^24
 * rows).
 * The caller allocates it; the library never does. */
size_t fckl_workspace_bytes(int64_t N, int d, int V, int K, int chunk, int dtype);

/* Bytes of a workspace with which fckl_forward_backward overlaps the steps of consecutive
 * chunks (same citation: at most two chunks' buffers are held, still independent of N beyond
 * the 4 bytes per position). With N > chunk this adds a second set of one chunk's buffers
 * (gradient slab, chunk * V * 2 bytes, and the chunk's ordered cache slots and tile
 * statistics) to fckl_workspace_bytes(); each chunk's G is then formed on a library-owned
 * second stream while the next chunk's forward runs on the caller's stream, and the caller's
 * stream waits for it before that chunk's gradient products, so the call still completes in
 * the caller's stream order and its results are bitwise those of the smaller workspace. The
 * library overlaps only where it pays: a projection of at least 5e11 FLOPs per chunk
 * (2 * chunk * d * V) and d >= 2048 (below that the G pass, at one block per SM beside the
 * forward, outlasts it); otherwise the chunks run in sequence. The environment variable
 * FCKL_OVERLAP=1 or 0 forces the choice. With N <= chunk it equals fckl_workspace_bytes().
 * 0 if the shape is outside the limits. */
size_t fckl_overlap_workspace_bytes(int64_t N, int d, int V, int K, int chunk, int dtype);

/* Forward pass ("Hugging Face：让知识蒸馏廉价到可大规模运行", paragraph "Fused, chunked KL
 * loss": each chunk's hidden states are projected to logits, folded into the accumulated loss
 * and dropped before the next chunk; paragraph "离线蒸馏": the loss is taken against the cached
 * top-100 tokens of every position; "Chunkovaná KL strata ...", section "Čo dopĺňajú
 * podrobnejšie experimenty": that truncated distribution is not renormalised, S_n < 1).
 * Per chunk: order the chunk's cache slots by id, then one tensor-core pass over the
 * vocabulary keeps, per row and 256-column tile, the tile maximum, the sum of exp(z - max) and
 * the sum of p z at the cached ids; no logit tile leaves the SM.
 *   loss     : device fp32 [1]  <- sum over positions of the per-position KL (a SUM, not a mean)
 *   lse      : device fp32 [N]  <- log-partition of every position, kept for fckl_backward
 *   row_loss : device fp32 [N]  <- per-position KL, or NULL when not wanted
 * Overwrites the workspace and clears its status word first. */
int fckl_forward(const void* H, const void* W, int dtype,
                 const int32_t* idx, const float* logp, const float* weight,
                 int64_t N, int d, int V, int K, int chunk,
                 float* loss, float* lse, float* row_loss,
                 void* ws, size_t ws_bytes, void* stream);

/* Backward pass ("Hugging Face：让知识蒸馏廉价到可大规模运行", paragraph "Fused, chunked KL
 * loss": the backward pass recomputes each chunk instead of storing it, so the projection runs
 * twice; the closing paragraph names the closed-form gradient, which is the derivative of the
 * loss above: G_n = S_n softmax(z_n) - p_sparse_n, dH = G W, dW = G^T H).
 * Recomputes every chunk's logits and forms G from `lse` (as written by
 * fckl_forward for the same H, W): per logit z with 256-column tile maximum m,
 * G = weight_n * grad_scale * (S_n exp(m - lse_n) e - p at the cached ids), e = exp(z - m)
 * rounded to fp16 (relative 2^-11), G rounded to bf16 (2^-9).
 *   grad_scale : upstream derivative d(objective)/d(loss); multiplies dH and dW
 *   dH         : device [N, d] of type `dtype`, overwritten
 *   dW         : device fp32 [V, d], overwritten
 * Overwrites the workspace and clears its status word first. */
int fckl_backward(const void* H, const void* W, int dtype,
                  const int32_t* idx, const float* logp, const float* weight, const float* lse,
                  int64_t N, int d, int V, int K, int chunk,
                  float grad_scale, void* dH, float* dW,
                  void* ws, size_t ws_bytes, void* stream);

/* Forward and backward in one call, chunk by chunk: each chunk's backward runs right after
 * its forward (lse_n depends on position n alone), so the chunk's cache slots are ordered
 * once and its hidden states are re-read while still in L2. Outputs as fckl_forward and
 * fckl_backward (row_loss may be NULL); the same workspace as the separate calls, or the
 * larger one of fckl_overlap_workspace_bytes (below).
 * The chunk's logits are not recomputed: its forward stores e = exp(z - m) as fp16 into the
 * gradient slab (m: the logit's 256-column tile maximum, kept with the softmax statistics)
 * and its backward turns the slab into G in place, G = S_n exp(m - lse_n) e - p at the cached
 * ids (times the weight and grad_scale). This saves one of the four products per chunk and
 * needs no memory beyond the slab. fckl_backward forms G from recomputed logits with the same
 * operations (tile maximum, fp16 e, the same products and roundings), so the two calls give
 * bitwise identical outputs. Not an operation of the pages' method: their backward recomputes
 * each chunk only because their forward drops it ("Fused, chunked KL loss"); here the backward
 * directly follows the forward. With ws_bytes >= fckl_overlap_workspace_bytes() and N > chunk,
 * consecutive chunks overlap: chunk c's G pass runs on the library's second stream beside chunk
 * c+1's forward, joined back into `stream` before chunk c's gradient products and before the
 * call returns; the outputs are bitwise those of the smaller workspace. */
int fckl_forward_backward(const void* H, const void* W, int dtype,
                          const int32_t* idx, const float* logp, const float* weight,
                          int64_t N, int d, int V, int K, int chunk, float grad_scale,
                          float* loss, float* lse, float* row_loss, void* dH, float* dW,
                          void* ws, size_t ws_bytes, void* stream);

/* Largest device scratch (bytes) that fckl_forward_static can use. The library reserves this
 * much device memory on every GPU where it is loaded, and keeps it until the process exits. */
#define FCKL_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* Forward pass that allocates nothing and takes no workspace.
 *
 * The pages have no counterpart to this call: it is an interface addition. It serves callers
 * that cannot allocate device memory at the point of the call, such as a custom operator or
 * plugin hosted by a framework or inference server that owns all device memory through its
 * own pool (a raw cudaMalloc there bypasses the pool and may fail once the pool holds the
 * memory), or a step loop where cudaMalloc/cudaFree and their synchronisation are not
 * acceptable. Such callers cannot hand fckl_forward a workspace, so this call uses a scratch
 * array of FCKL_STATIC_SCRATCH_BYTES that the library itself keeps in device memory.
 *
 * Inputs and outputs are those of fckl_forward (bf16 H and W only; dtype must be FCKL_BF16),
 * except that row_loss is required (the loss sum reads it) and
 *   status : device uint32 [1] <- status bits found on the device by this call
 *            (0 = clean, bit 0 = a teacher id outside [0, V), bit 1 = a device wait ran out)
 * The scratch needed is about (8*K + 8 + 12*ceil(V/256)) bytes per row of a chunk rounded up to
 * 256 rows; a shape above FCKL_STATIC_SCRATCH_BYTES is rejected with FCKL_ERR_WORKSPACE and a
 * message in fckl_last_error(), before anything is launched. At K = 100 and V = 128256 a chunk
 * of up to 4096 positions fits.
 *
 * The first call on a device looks up the device address of the array (cudaGetSymbolAddress
 * with that device current); make that first call before any stream capture. Later calls look
 * the address up again unless their stream is being captured (then the address of the last
 * uncaptured call on that device is used), so a device reset or another context of the same
 * device gets the array's current address.
 * Every call on a device shares the one array, which keeps the previous call's contents (the
 * call clears the status word it needs zeroed): calls whose work overlaps on the GPU (on
 * different streams, or from different threads) race on it and must be serialised by the
 * caller. The call calls no cudaMalloc, cudaFree or other allocating routine. */
int fckl_forward_static(const void* H, const void* W, int dtype,
                        const int32_t* idx, const float* logp,
                        int64_t N, int d, int V, int K, int chunk,
                        float* loss, float* lse, float* row_loss,
                        uint32_t* status, void* stream);

/* Offline teacher top-K cache ("Hugging Face：让知识蒸馏廉价到可大规模运行", paragraph "离线蒸馏":
 * the teacher runs once and the 100 most probable tokens of every position are cached;
 * "Chunkovaná KL strata ...", section "Čo dopĺňajú podrobnejšie experimenty": kept without
 * renormalisation). For every position n of the teacher hidden states Ht [N, d] and output
 * matrix Wt [V, d] (dtype as for the loss), writes the K token ids of largest logit
 * z_nv = Wt_v . h_n and their log-probabilities under the full softmax, z_nv - lse_n:
 *   idx  : device int32 [N, K], each row ordered by logit descending, equal logits by smaller id
 *   logp : device fp32  [N, K]
 * Two passes per chunk: the first projects the chunk and keeps each row's per-tile maxima and
 * sum-exp (giving lse_n and a threshold, the K-th largest tile maximum, that every top-K
 * logit reaches); the second keeps the logits at or above the threshold as candidates, which
 * are then ranked exactly. The second pass reads the chunk's logits as the first pass stored
 * them when ws_bytes >= fckl_topk_kept_logits_workspace_bytes() (4 * chunk * V bytes more),
 * else it projects the chunk again; the outputs are the same either way. With ws_bytes >=
 * fckl_topk_overlap_workspace_bytes() (a second set of one chunk's kept logits, candidates and
 * per-row values) and N > chunk, each chunk's second pass and ranking run on the library's
 * second stream (as in fckl_forward_backward) beside the next chunk's first pass, joined back
 * into `stream` before the call returns, when the first pass is at least 5e11 FLOPs per chunk
 * (FCKL_OVERLAP=1 or 0 forces the choice); the outputs are again the same. A row with more
 * candidates than the buffer holds (min(V, 2048) slots, or V when K exceeds ceil(V/256)) is
 * reported as FCKL_ERR_CAPACITY by fckl_check. The workspace is at least
 * fckl_topk_workspace_bytes. V up to 1,310,720 (FCKL_ERR_UNSUPPORTED above). */
size_t fckl_topk_workspace_bytes(int64_t N, int d, int V, int K, int chunk, int dtype);
size_t fckl_topk_kept_logits_workspace_bytes(int64_t N, int d, int V, int K, int chunk, int dtype);
size_t fckl_topk_overlap_workspace_bytes(int64_t N, int d, int V, int K, int chunk, int dtype);
int fckl_teacher_topk(const void* Ht, const void* Wt, int dtype,
                      int64_t N, int d, int V, int K, int chunk,
                      int32_t* idx, float* logp,
                      void* ws, size_t ws_bytes, void* stream);

/* Interface addition, no counterpart on the pages (they describe no device interface).
 * Synchronises `stream`, returns the status found on the device by the last call that
 * used `ws` (FCKL_OK if none), and clears it. */
int fckl_check(void* ws, void* stream);

/* Interface addition, no counterpart on the pages.
 * Self-test of failure detection: launches one kernel that waits, with the same bounded
 * wait the pipeline kernels use but a 50 ms limit, on a barrier nothing arrives at. The wait
 * gives up, the kernel records a timeout in the status word at the start of ws and returns
 * normally, so fckl_check(ws, stream) then returns FCKL_ERR_TIMEOUT and the context stays
 * usable. ws: device buffer of at least 256 bytes (any fckl workspace will do). */
int fckl_selftest_wait_timeout(void* ws, size_t ws_bytes, void* stream);

/* Diagnostics below: interface additions, no counterpart on the pages.
 * Static text for a status code. */
const char* fckl_status_string(int status);

/* Text of the last CUDA error seen by this library in this process ("" if none). */
const char* fckl_last_error(void);

/* Number of kernels this library has launched in this process. */
int64_t fckl_launch_count(void);

/* Per-kernel timing. While enabled, every launch is bracketed by CUDA events recorded on
 * its own stream. fckl_profile_read synchronises the device, adds the measured time (ms)
 * and launch count of each kernel kind into ms[kind] and launches[kind] for kind <
 * n_kinds, and forgets the events. fckl_kernel_name(kind) names a kind (NULL past the
 * last). */
int fckl_profile_enable(int on);
int fckl_profile_read(double* ms, int64_t* launches, int n_kinds);
const char* fckl_kernel_name(int kind);

#ifdef __cplusplus
}
#endif

#endif /* FCKL_H */

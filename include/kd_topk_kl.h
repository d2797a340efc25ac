/*
 * kd_topk_kl.h -- C ABI of the fused chunked top-K KL distillation loss
 * (forward + backward) for NVIDIA B300 (sm_103a).
 *
 * The operation.  Multiverse Computing, "Efficient Knowledge Distillation for
 * LLMs: Offline Top-K Logits and a Fused Chunked KL Loss", as described on
 * its news coverage:
 *   - the teacher's K highest logits and their token ids are computed once,
 *     offline, and stored per position (epoka.news, "The two proposed
 *     changes"; ainewsbank.com, "Two changes remove different bottlenecks":
 *     K = 100 there);
 *   - the loss handles the token positions chunk by chunk: a chunk's
 *     logits are formed, reduced into the running loss and dropped, then
 *     formed again during the backward pass rather than kept (glonce.com,
 *     body, the paragraph on Multiverse's fix), so no [tokens x vocab]
 *     logit matrix ever exists in memory (glonce.com, "Key facts").
 * The pages do not print the formula.  This library computes the standard
 * truncated-teacher KL, with z_n = W h_n (no bias), T > 0:
 *   p_nk    = softmax_k(topk_logit_n / T)              over the K entries
 *   log q_nv = z_nv / T - logsumexp_v(z_n / T)          over all V
 *   loss    = (1/N) sum_n sum_k p_nk (log p_nk - log q_{n, idx_nk})
 *   dZ_nv   = (q_nv - sum_{k: idx_nk = v} p_nk) / (T N)
 *   grad_hidden = dZ W,  grad_W = dZ^T hidden
 * There is no T^2 factor; the mean is over all N tokens; repeated ids add
 * up in dZ and give one loss term each.
 *
 * Arithmetic.  hidden and W are bf16; the GEMMs run on tcgen05 tensor cores
 * with fp32 accumulation; each token's logsumexp and dot product with the
 * teacher are fp32, its loss term is combined and the terms summed in
 * double; dZ is held as bf16 scratch for two consecutive chunks
 * (2 x chunk x V; one chunk with KD_FLAG_MIN_SCRATCH); grad_W is
 * accumulated over those chunk pairs in fp32 in device memory.
 *
 * Pointers.  Unless stated otherwise every array argument is a DEVICE
 * pointer (cudaMalloc / cudaMallocAsync / managed memory on the current
 * device) owned by the caller; the library never frees or keeps it.  Host or
 * unregistered pointers are rejected with KD_ERR_INVALID_ARG before any
 * launch.  All arrays are dense and row-major.
 *
 * Pointers to device memory must belong to the current device (managed
 * memory is accepted too).
 *
 * Errors.  Argument errors are detected on the host before anything is
 * launched.  Device-side errors (an id outside [0, V), a bounded wait that
 * ran out) are reported after the stream has been synchronised; on any
 * error the outputs are unspecified.  Every call except
 * kd_topk_kl_fwd_bwd_async returns after a stream synchronisation (also
 * after a CUDA error part-way through), because `loss` is a host pointer:
 * when it returns, none of its kernels still uses the workspace or the
 * outputs.  kd_topk_kl_fwd_bwd_async leaves the loss and the device-side
 * status in device memory and does not wait (see there).
 *
 * Thread safety.  Calls on different streams may run concurrently, from one
 * host thread or several, if they use different workspaces and outputs; they
 * give bitwise the results of the same calls run one after another.  A call
 * uses the calling thread's current device; if no context is current on the
 * thread it makes the device's primary context current (a context the caller
 * made current is left in place).  The profiler (kd_profile_*) and the
 * no-alloc entry point's shared buffer are the exceptions (see there).
 */
#ifndef KD_TOPK_KL_H
#define KD_TOPK_KL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kd_status {
  KD_OK = 0,
  KD_ERR_INVALID_ARG = 1,     /* a size, a null pointer, a host pointer, T <= 0 ... */
  KD_ERR_ALIGNMENT = 2,       /* a base pointer not aligned as documented */
  KD_ERR_INDEX = 3,           /* some topk_idx entry lies outside [0, V) */
  KD_ERR_OOM = 4,             /* workspace allocation failed / too small */
  KD_ERR_CUDA = 5,            /* a CUDA runtime error; see kd_last_cuda_error() */
  KD_ERR_TIMEOUT = 6,         /* a bounded device-side wait ran out */
  KD_ERR_NOT_IMPLEMENTED = 7,
  KD_ERR_TOO_LARGE = 8        /* kd_topk_kl_fwd_bwd_noalloc: the problem's scratch exceeds
                                 KD_NOALLOC_SCRATCH_BYTES */
} kd_status;

/*
 * Loss and gradients of the top-K KL loss, using the legacy default stream
 * and a workspace the call allocates (stream-ordered) and frees itself.
 *
 *   hidden      bf16 [N, H]  student final hidden states (device)
 *   W           bf16 [V, H]  LM-head weight, z = hidden W^T (device)
 *   topk_idx    int32 [N, K] cached teacher token ids, in [0, V) (device)
 *   topk_logit  fp32 [N, K]  cached teacher logits, paired with topk_idx
 *   N           tokens, 1 <= N <= 2^31 - 1
 *   H           hidden size, H % 8 == 0
 *   V           vocabulary size, V % 8 == 0, V <= 2^31 - 1
 *   K           cached entries per token, 1 <= K <= min(V, 8192)
 *   T           temperature, finite and > 0
 *   chunk       token rows per chunk (>= 1); rounded up to a multiple of 128
 *               and capped at N rounded up likewise, and at 2^30 rows.
 *               Scratch grows as 2 x chunk x V x 2 bytes (the bf16 dZ of
 *               two chunks; one chunk's when N fits in one chunk).
 *   loss        HOST float*: the mean over the N tokens
 *   grad_hidden fp32 [N, H] (device), overwritten
 *   grad_W      fp32 [V, H] (device), overwritten
 *
 * Alignment: hidden, W, grad_hidden and grad_W 16-byte aligned; topk_idx
 * and topk_logit 4-byte aligned.  Ids are not checked for distinctness;
 * repeated ids follow the scatter-add reading above.
 */
kd_status kd_topk_kl_fwd_bwd(const void* hidden, const void* W, const int32_t* topk_idx,
                             const float* topk_logit, int64_t N, int H, int V, int K, float T,
                             int chunk, float* loss, float* grad_hidden, float* grad_W);

/*
 * Bytes of device workspace kd_topk_kl_fwd_bwd_ex needs for these sizes on
 * the CURRENT device (the split of one GEMM depends on its SM count).
 * Returns 0 when the sizes are invalid.
 */
size_t kd_topk_kl_workspace_size(int64_t N, int H, int V, int K, int chunk);

/*
 * As kd_topk_kl_fwd_bwd, on the caller's stream and with a caller-owned
 * workspace of at least kd_topk_kl_workspace_size(...) bytes, 256-byte
 * aligned (device).  `stream` is a cudaStream_t (NULL = legacy default
 * stream).  The workspace's contents on entry do not matter; it must not be
 * used by anything else until the call returns.
 */
kd_status kd_topk_kl_fwd_bwd_ex(const void* hidden, const void* W, const int32_t* topk_idx,
                                const float* topk_logit, int64_t N, int H, int V, int K, float T,
                                int chunk, float* loss, float* grad_hidden, float* grad_W,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * kd_topk_kl_fwd_bwd_ex with a per-token mask and an accumulate flag, for a
 * training step with padding or sequence packing (the pages mention packing
 * ablations only: glonce.com, body and "How to use it").
 *
 *   token_mask  uint8 [N] (device) or NULL.  Nonzero = the token counts.  The
 *               loss is the mean over the N_v valid tokens,
 *                 loss = (1/N_v) sum_{n valid} sum_k p_nk (log p_nk - log q_{n,idx_nk}),
 *               a masked token contributes no loss and zero gradient rows,
 *               and dZ is scaled by 1/(T N_v).  N_v = 0 gives loss 0 and zero
 *               gradients.  NULL = every token counts (same as _ex).
 *               Masked tokens' ids are still range-checked.
 *   accumulate  nonzero: grad_hidden += and grad_W += the call's gradients
 *               (both must hold finite values on entry); 0: overwrite.
 * Every other argument as for kd_topk_kl_fwd_bwd_ex.
 */
kd_status kd_topk_kl_fwd_bwd_masked(const void* hidden, const void* W, const int32_t* topk_idx,
                                    const float* topk_logit, const uint8_t* token_mask,
                                    int64_t N, int H, int V, int K, float T, int chunk,
                                    int accumulate, float* loss, float* grad_hidden,
                                    float* grad_W, void* workspace, size_t workspace_bytes,
                                    void* stream);

/* Flags of kd_topk_kl_fwd_bwd_flags / kd_topk_kl_workspace_size_flags. */
#define KD_FLAG_ACCUMULATE 1u     /* add into grad_hidden / grad_W instead of overwriting */
#define KD_FLAG_STORE_LOGITS 2u   /* keep each chunk's logits between forward and backward */
#define KD_FLAG_MIN_SCRATCH 4u    /* one chunk's dZ in the workspace instead of two (see below) */

/*
 * Workspace bytes for kd_topk_kl_fwd_bwd_flags with these flags (0 when the
 * sizes or the flags are invalid).  KD_FLAG_STORE_LOGITS adds chunk x V x 4
 * bytes (the chunk's fp32 logits).
 *
 * By default a call with two or more chunks keeps the bf16 dZ of two
 * consecutive chunks (2 x chunk x V x 2 bytes) and forms grad_W once per
 * pair of chunks, reducing over both chunks' rows at once: the fp32
 * read-modify-write of all of grad_W (V x H x 8 bytes) then happens once per
 * two chunks instead of once per chunk.  KD_FLAG_MIN_SCRATCH keeps one
 * chunk's dZ (chunk x V x 2 bytes) and forms grad_W per chunk.  Both give
 * the same result up to the fp32 rounding of grad_W's accumulation order.
 */
size_t kd_topk_kl_workspace_size_flags(int64_t N, int H, int V, int K, int chunk,
                                       unsigned flags);

/*
 * kd_topk_kl_fwd_bwd_masked with flags.
 *
 * KD_FLAG_STORE_LOGITS is an ablation of the recompute the pages describe
 * (glonce.com, body: the fused loss recomputes chunks during the backward
 * pass instead of storing them, and at 8K context that extra projection
 * costs some speed).  The forward GEMM also writes the chunk's fp32 logits
 * to the workspace, and the backward forms dZ from them with an elementwise
 * kernel instead of recomputing the GEMM: 6 N H V instead of 8 N H V flops,
 * for chunk x V x 4 more bytes of workspace.  The logits are the very values
 * the recompute would produce, and dZ is rounded the same way, so the
 * results are bitwise those of the recompute path.
 */
kd_status kd_topk_kl_fwd_bwd_flags(const void* hidden, const void* W, const int32_t* topk_idx,
                                   const float* topk_logit, const uint8_t* token_mask,
                                   int64_t N, int H, int V, int K, float T, int chunk,
                                   unsigned flags, float* loss, float* grad_hidden, float* grad_W,
                                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * One shard of a batch whose loss is the mean over n_norm tokens.
 *
 * The pages' headline run distils GPT-OSS 20B at 32K context on one node
 * instead of four (glonce.com, body and "Key facts"); a data-parallel
 * trainer splits a batch's tokens across devices, and a single-device
 * trainer may split them into micro-batches.  Both need each shard's loss
 * and gradients normalised by the whole batch's token count, so that the
 * shards' results add up:
 *
 *   loss (out)   (1/n_norm) sum over this shard's (valid) tokens of the
 *                per-token KL terms; the batch loss is the sum over shards
 *   grad_hidden  this shard's rows, scaled by 1/(T n_norm): final as they are
 *   grad_W       this shard's share, scaled by 1/(T n_norm); the batch's
 *                grad_W is the sum of the shards' (add them with
 *                KD_FLAG_ACCUMULATE on one device, or an all-reduce across
 *                devices).  KD_FLAG_ACCUMULATE adds into grad_hidden too: a
 *                shard that accumulates grad_W needs its grad_hidden rows
 *                to hold zeros (or what they should be added to) on entry
 *   n_norm       >= 1: the number of tokens the batch's mean runs over (with
 *                masks, the batch's valid tokens); KD_ERR_INVALID_ARG otherwise
 *
 * Everything else as for kd_topk_kl_fwd_bwd_flags (N, hidden, topk_* and
 * token_mask describe the shard).  With n_norm = N (or N_v for a masked
 * call) the results equal kd_topk_kl_fwd_bwd_flags's.
 */
kd_status kd_topk_kl_fwd_bwd_sharded(const void* hidden, const void* W, const int32_t* topk_idx,
                                     const float* topk_logit, const uint8_t* token_mask,
                                     int64_t N, int H, int V, int K, float T, int chunk,
                                     unsigned flags, int64_t n_norm, float* loss,
                                     float* grad_hidden, float* grad_W, void* workspace,
                                     size_t workspace_bytes, void* stream);

/*
 * Asynchronous form of kd_topk_kl_fwd_bwd_flags, for a training step that
 * keeps the host out of the loop or captures the step in a CUDA graph.  It
 * enqueues the whole path on `stream` and returns without synchronising:
 *
 *   loss_dev    fp32 [1] (device): the loss, as kd_topk_kl_fwd_bwd_flags
 *               would return it (the same float, bit for bit)
 *   status_dev  int32 [1] (device): KD_OK, KD_ERR_INDEX (an id outside
 *               [0, V)) or KD_ERR_TIMEOUT (a bounded wait ran out), written
 *               by the call's last kernel
 *
 * Both are valid once the stream has reached the end of the call; the
 * gradients are valid when *status_dev == KD_OK.  The return value covers
 * only what the host checks before anything is enqueued (arguments,
 * workspace size, alignment) and CUDA errors while enqueuing; on any return
 * other than KD_OK nothing of the call needs to be waited for, except after
 * KD_ERR_CUDA, when the caller synchronises the stream before reusing the
 * buffers (outside a graph capture the call does so itself).
 *
 * Every operation the call enqueues is a kernel launch or a memset on
 * `stream`, and the TMA descriptors travel by value in the launch
 * parameters, so the call may be captured into a CUDA graph.  A replay
 * reuses the pointers and sizes of the capture: new inputs are written into
 * the same buffers.  The library's per-kernel profiler does not time this
 * call.  The workspace and both device words belong to the call until the
 * stream has passed it.  Every other argument as for
 * kd_topk_kl_fwd_bwd_flags.
 */
kd_status kd_topk_kl_fwd_bwd_async(const void* hidden, const void* W, const int32_t* topk_idx,
                                   const float* topk_logit, const uint8_t* token_mask,
                                   int64_t N, int H, int V, int K, float T, int chunk,
                                   unsigned flags, float* loss_dev, int32_t* status_dev,
                                   float* grad_hidden, float* grad_W, void* workspace,
                                   size_t workspace_bytes, void* stream);

/*
 * The offline top-K teacher cache (the step before the loss): per token,
 * the teacher's K highest logits and their ids, computed once and stored
 * (epoka.news, "The two proposed changes"; glonce.com, body;
 * ainewsbank.com, "Two changes remove different bottlenecks": K = 100).
 *
 *   hidden      bf16 [N, H]  teacher final hidden states (device)
 *   W           bf16 [V, H]  teacher LM head, z = hidden W^T (device)
 *   K           1 <= K <= min(V, 8192)
 *   chunk       token rows per chunk (rounded up to a multiple of 128); the
 *               workspace holds one chunk's fp32 logits (chunk x V x 4 bytes)
 *               and a 16 KB candidate list per row of the chunk
 *   topk_idx    int32 [N, K] out (device): ids in decreasing logit order,
 *               equal logits in increasing id order (the pages leave ties open)
 *   topk_logit  fp32 [N, K] out (device): the logits z (fp32 accumulation of
 *               the bf16 products), decreasing
 * The logits are computed on the tensor cores one chunk at a time; the
 * selection is exact for those fp32 values.  Same pointer, error and
 * synchronisation rules as kd_topk_kl_fwd_bwd_ex; the caller owns the
 * workspace (kd_topk_cache_workspace_size bytes, 256-byte aligned).
 */
size_t kd_topk_cache_workspace_size(int64_t N, int H, int V, int K, int chunk);
kd_status kd_topk_cache_build(const void* hidden, const void* W, int64_t N, int H, int V, int K,
                              int chunk, int32_t* topk_idx, float* topk_logit, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * Test and diagnosis options for kd_topk_kl_debug.  Each output pointer may
 * be NULL (not written).
 *   lse        fp32 [N]    logsumexp_v(z_n / T) (device)
 *   zg         fp32 [N, K] z at topk_idx, in the caller's k order (device)
 *   found_idx  int32 [N, K] the vocabulary column at which the forward
 *              epilogue met topk_idx[n, k]; must be pre-filled by the caller
 *              (e.g. with -1) -- it equals topk_idx exactly when every id
 *              was gathered from the right column (device)
 *   loss_rows  double [N] the per-token terms sum_k p (log p - log q_idx),
 *              whose mean is the loss (device)
 *   timeout_ns limit of every device-side wait (0 = the default, 5 s)
 *   inject_timeout  1 / 2 / 3 / 4: the first chunk's forward / recompute /
 *              grad_hidden / grad_W GEMM's epilogue waits on a barrier
 *              that nothing completes, so the call must end with
 *              KD_ERR_TIMEOUT after ~timeout_ns without hanging
 */
typedef struct kd_debug_opts {
  float* lse;
  float* zg;
  int32_t* found_idx;
  uint64_t timeout_ns;
  int inject_timeout;
  double* loss_rows;
} kd_debug_opts;

/* kd_topk_kl_fwd_bwd_ex plus the exports and hooks of `opts` (may be NULL). */
kd_status kd_topk_kl_debug(const void* hidden, const void* W, const int32_t* topk_idx,
                           const float* topk_logit, int64_t N, int H, int V, int K, float T,
                           int chunk, float* loss, float* grad_hidden, float* grad_W,
                           void* workspace, size_t workspace_bytes, void* stream,
                           const kd_debug_opts* opts);

/*
 * Test entry of the tensor-core GEMM core alone (no paper counterpart; it
 * checks the operand layouts the loss uses):  C = A * B^T with
 *   A  bf16, [M, K] when a_mn == 0 (K contiguous) or [K, M] when a_mn != 0
 *   B  bf16, [N, K] when b_mn == 0 or [K, N] when b_mn != 0
 *   C  fp32 [M, N]
 * pair == 0: one CTA per 128 x bn tile, bn the tile width of the N dimension
 * (192 or 256; 0 = the default of this layout).  pair != 0: a CTA pair per
 * 256 x 256 tile with 2-CTA MMAs, the form the loss's GEMMs use (bn 0 or
 * 256); pair == 2: the same with two 64-deep k-blocks per pipeline stage
 * (K-major A and B only).  M, N, K multiples of 8; all pointers device,
 * 16-byte aligned.
 * Synchronises `stream` before returning.
 */
kd_status kd_gemm_bf16_test(const void* A, const void* B, float* C, int M, int N, int K, int a_mn,
                            int b_mn, int bn, int pair, void* stream);

/*
 * Per-kernel timing (diagnostics; no paper counterpart).  While enabled,
 * every kernel launch of kd_topk_kl_fwd_bwd[_ex] / kd_topk_kl_debug is
 * bracketed by two CUDA events on the call's stream, and after the call's
 * final synchronisation the elapsed times are added to per-kind totals.
 * kd_profile_enable(1) resets the totals; kd_profile_enable(0) stops.
 * kd_profile_read fills up to max_kinds entries of total_ms (milliseconds)
 * and launches (either may be NULL) and returns the number of kinds;
 * kd_profile_kind_name names kind i.  Process-global: not for concurrent
 * calls from several threads.
 */
void kd_profile_enable(int on);
int kd_profile_read(double* total_ms, long long* launches, int max_kinds);
const char* kd_profile_kind_name(int kind);

/*
 * Size of the library's built-in scratch buffer used by
 * kd_topk_kl_fwd_bwd_noalloc (64 MiB on each device, from the first call
 * on that device until the process exits).
 */
#define KD_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * kd_topk_kl_fwd_bwd without any allocation (no paper counterpart).
 *
 * For callers that cannot allocate device memory on their own: code running
 * where a cudaMalloc / cudaMallocAsync (or a framework allocator) is not
 * permitted or not available, e.g. a host framework that owns every
 * allocation, or a runtime that has already reserved all memory for its own
 * pool.  The caller still provides the inputs and outputs exactly as for
 * kd_topk_kl_fwd_bwd_ex; the call's workspace is a fixed buffer compiled
 * into the library (KD_NOALLOC_SCRATCH_BYTES, 64 MiB per device).
 *
 *  - Sizes whose kd_topk_kl_workspace_size() exceeds KD_NOALLOC_SCRATCH_BYTES
 *    are rejected with KD_ERR_TOO_LARGE before anything is launched.  The
 *    scratch grows with chunk x V (the bf16 dZ of one chunk, or of two when
 *    the call has two chunks or more) and N x K (the sorted teacher tables);
 *    for example N = 4096, H = 4096, V = 32,000, K = 100 fits at chunk 128
 *    (about 41 MiB), while a 201,088-token vocabulary at chunk 128 and 4,096
 *    tokens does not.
 *  - The first call on a device looks up the buffer's device address on the
 *    current device (cudaGetSymbolAddress); make that first call before any
 *    stream capture.  CUDA loads a library's device code, and with it this
 *    buffer, when it is first used on a device, so the 64 MiB are taken
 *    from the device at that first call: a caller whose memory pool will
 *    take the rest of the device makes one call (any valid size) before the
 *    pool reserves it.  If the device cannot hold the buffer then, the call
 *    returns KD_ERR_OOM.
 *  - The buffer is shared by every call on a device and keeps the previous
 *    call's contents; each call resets what must start at zero.  Calls whose
 *    work overlaps on the GPU (several streams or threads at once) race on
 *    the buffer and give wrong results: serialise them.
 *  - No cudaMalloc, cudaFree or allocating routine is called.  Like
 *    kd_topk_kl_fwd_bwd_ex it synchronises `stream` (a cudaStream_t, NULL =
 *    legacy default stream) before returning.
 */
kd_status kd_topk_kl_fwd_bwd_noalloc(const void* hidden, const void* W, const int32_t* topk_idx,
                                     const float* topk_logit, int64_t N, int H, int V, int K,
                                     float T, int chunk, float* loss, float* grad_hidden,
                                     float* grad_W, void* stream);

/* Static text for a status code. */
const char* kd_status_string(kd_status s);

/* Text of the last CUDA error this library saw on the calling thread ("" if none). */
const char* kd_last_cuda_error(void);

/* Version of this ABI (incremented on any incompatible change). */
int kd_abi_version(void);

/* Identity of the sources this library was built from: the first 16 hex
 * digits of a SHA-256 over the CUDA sources, this header and the build
 * script, fixed at compile time ("unknown" for a build that did not set
 * it).  Static text. */
const char* kd_build_id(void);

#ifdef __cplusplus
}
#endif

#endif /* KD_TOPK_KL_H */

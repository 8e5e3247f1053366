/*
 * libpath_attn — PaTH attention on one NVIDIA GB300 (sm_103a).
 *
 * PaTH attention (PaTH Attention summary, gist.science/ko/paper/2505.16381,
 * section "2. 방법론 / 핵심 메커니즘", attention-logit equation) is causal
 * softmax attention whose logit between query i and key j <= i is
 *
 *     scale * k_j^T (H_{j+1} H_{j+2} ... H_i) q_i,    H_s = I - beta_s w_s w_s^T,
 *
 * with one unit direction w_s and one coefficient beta_s in [0, 2] per token
 * and head.  The product is ordered so that H_i acts on q_i first; for
 * j == i it is the identity.  PaTH-FoX (section "확장: PaTH-FoX") adds the
 * forgetting-transformer bias sum_{s=j+1}^{i} log f_s, unscaled.
 *
 * Conventions shared by every call:
 *   - Tensors are dense, row-major, on the current CUDA device.  Activations
 *     q, k, v, w, out are [batch][heads][seq_len][head_dim]; beta, log_f and
 *     lse are float32 [batch][heads][seq_len].  The element type of q, k, v,
 *     w, out and the caches is the descriptor's dtype.
 *   - Every device pointer must be 16-byte aligned.
 *   - The caller owns every buffer, the workspace included.  The library
 *     allocates no memory and keeps no state between calls, besides a
 *     one-word device error flag (see path_attn_device_status) and the fixed
 *     scratch array of path_attn_decode_step_noalloc.
 *   - Calls are asynchronous on `stream`.  Argument errors are returned
 *     before anything is launched.  A launch failure returns PATH_ERR_CUDA.
 *   - Preconditions the library does not check or enforce: w rows have unit
 *     norm and beta lies in [0, 2]; nothing is normalised or clipped.
 *   - Calls that overlap in time on the GPU must not share a workspace.
 */
#ifndef PATH_ATTN_H
#define PATH_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* A cudaStream_t.  NULL selects the legacy default stream. */
typedef struct CUstream_st *path_stream_t;

typedef enum {
    PATH_OK = 0,
    PATH_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or workspace   */
    PATH_ERR_UNSUPPORTED = 2, /* valid but not implemented (dtype, head_dim) */
    PATH_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed        */
    PATH_ERR_TIMEOUT = 4      /* a device-side wait hit its iteration limit  */
} path_status_t;

typedef enum { PATH_F32 = 0, PATH_BF16 = 1 } path_dtype_t;

/* ------------------------------------------------------------------ prefill */

typedef struct {
    int32_t batch, heads, seq_len, head_dim;
    int32_t dtype;  /* path_dtype_t */
    float scale;    /* multiplies k^T(...)q; usually 1/sqrt(head_dim) */
    int32_t chunk;  /* 0 = default. PATH_BF16 with head_dim 128: 128 only
                       (head_dim a multiple of 8 below 128: 0 or 128 for the
                       tensor cores, others on the CUDA cores).
                       Otherwise 16, 32, 64 or 128; the default is 64
                       when batch*heads*seq_len <= 8192 and head_dim <= 64,
                       else 128. */
    int32_t scan_group; /* tensor-core scan only: heads per group of its
                           tile order (the query tiles of one group of heads
                           are handed out, heaviest first, before the next
                           group's).  0 = automatic: about SM count / 10 heads
                           (at least 2.5 grids of tiles per group), groups of
                           equal size.  Values above batch*heads mean one
                           group.  It changes only the speed, never a result.
                           Negative: PATH_ERR_INVALID_ARG. */
} path_prefill_desc_t;

/*
 * Bytes of device workspace path_attn_prefill_fwd needs for `desc` (0 if the
 * descriptor is invalid).  The workspace holds, per head, the
 * boundary-adjusted query and key rows, the chunk products in compact form
 * and the within-chunk logits (section "3. 효율적인 학습 및 추론",
 * FlashAttention-style algorithm); its contents are unspecified between
 * calls.
 */
size_t path_attn_prefill_workspace_size(const path_prefill_desc_t *desc);

/*
 * Causal PaTH (or PaTH-FoX) attention forward.
 *   q, k, v, w : [B][H][L][d], desc->dtype.
 *   beta       : float32 [B][H][L].
 *   log_f      : float32 [B][H][L] log forget gate (PaTH-FoX), or NULL.
 *   out        : [B][H][L][d], desc->dtype, written.
 *   lse        : float32 [B][H][L], natural log of the sum of exp(logit) over
 *                the causal row (logits include scale and FoX bias), or NULL.
 *   workspace  : device buffer of at least
 *                path_attn_prefill_workspace_size(desc) bytes.
 * Supported: head_dim <= 128 and a multiple of 4, PATH_F32 or PATH_BF16.
 * PATH_BF16 with head_dim 128 runs on the tensor cores (chunk 128); so does
 * PATH_BF16 with head_dim a multiple of 8 below 128 and chunk 0 or 128, on
 * copies zero-padded to 128 in the workspace (exact: the padded coordinates
 * do not change any logit).  Every other case runs on the CUDA cores in fp32
 * (bf16 inputs and output converted on load and store).  seq_len may be any value >= 1 (the last
 * chunk may be partial).  Method: section 3 of the PaTH summary — a per-chunk UT
 * transform builds boundary-adjusted rows and the compact chunk product,
 * then a blockwise scan visits key chunks right to left, carrying the
 * accumulated product on the query side, with an online softmax.
 */
path_status_t path_attn_prefill_fwd(const path_prefill_desc_t *desc, const void *q,
                                    const void *k, const void *v, const void *w,
                                    const float *beta, const float *log_f, void *out,
                                    float *lse, void *workspace, size_t workspace_bytes,
                                    path_stream_t stream);

/*
 * The two stages of path_attn_prefill_fwd, callable separately (same
 * descriptor, same workspace; prefill_fwd computes exactly prep then scan,
 * with identical results; inside prefill_fwd the scan may start on the SMs
 * the prep has left while the prep's last chunks run, each of its query
 * tiles waiting until the prep has finished that tile's head):
 *
 * path_attn_prefill_prep: per chunk, the UT transform of the chunk's
 * transitions and everything derived from it (boundary-adjusted rows, the
 * chunk product, the chunk's own causal attention block), plus the FoX
 * prefix sums when log_f != NULL; written into the workspace.
 *
 * path_attn_prefill_scan: the right-to-left blockwise scan with online
 * softmax over the prep results; w and v are the same tensors given to the
 * prep call's problem; log_f must be non-NULL exactly when it was for the
 * prep call (only its presence is used here).
 */
path_status_t path_attn_prefill_prep(const path_prefill_desc_t *desc, const void *q,
                                     const void *k, const void *v, const void *w,
                                     const float *beta, const float *log_f, void *workspace,
                                     size_t workspace_bytes, path_stream_t stream);
path_status_t path_attn_prefill_scan(const path_prefill_desc_t *desc, const void *w,
                                     const void *v, const float *log_f, void *out, float *lse,
                                     void *workspace, size_t workspace_bytes,
                                     path_stream_t stream);

/* ----------------------------------------------------------------- backward */

/* Workspace of path_attn_prefill_bwd (0 if the descriptor is invalid).
 *
 * path_attn_prefill_bwd_workspace_size: the bytes to run every (batch, head)
 * slice in one pass, the fastest.  It grows as
 * batch*heads*seq_len^2*head_dim/chunk: per slice the backward keeps the
 * carried query rows of every (query chunk, earlier key chunk) pair (bf16 on
 * the tensor-core route, fp32 on the CUDA cores).
 *
 * path_attn_prefill_bwd_workspace_min: the bytes for one slice per pass, the
 * least path_attn_prefill_bwd accepts.  Any workspace in between works: the
 * call then runs the slices in passes of as many as the workspace holds, so
 * its size is the caller's choice between memory and speed (for example
 * about 1 GB at batch 8, 12 heads, 4096 positions, head_dim 128, 16 slices
 * per pass, against 6.4 GB in one pass). */
size_t path_attn_prefill_bwd_workspace_size(const path_prefill_desc_t *desc);
size_t path_attn_prefill_bwd_workspace_min(const path_prefill_desc_t *desc);

/*
 * Backward of path_attn_prefill_fwd: the gradients of
 *     sum(dout * out) + sum(dlse * lse)
 * with respect to q, k, v, w, beta and (PaTH-FoX) log_f.  The pages give no
 * backward algorithm; this one is reverse-mode differentiation of the
 * forward's blockwise algorithm (section 3 of the PaTH summary), recomputing
 * the per-chunk UT transform and re-walking the scan, with the per-key-chunk
 * sums accumulated atomically across query chunks.
 *   q, k, v, w   : the forward's inputs; beta, log_f likewise (log_f NULL for PaTH).
 *   out, lse     : the forward's outputs for these inputs (lse is required).
 *   dout         : [B][H][L][d], desc->dtype.
 *   dlse         : float32 [B][H][L], or NULL for zero.
 *   dq, dk, dv, dw : [B][H][L][d], desc->dtype, written.
 *   dbeta        : float32 [B][H][L], written.
 *   dlog_f       : float32 [B][H][L], written; required exactly when log_f is given.
 *   workspace    : at least path_attn_prefill_bwd_workspace_min(desc) bytes
 *                  (see above; path_attn_prefill_bwd_workspace_size(desc) for
 *                  one pass).
 * PATH_BF16 with head_dim 128 and chunk 128 (the default there) runs on the
 * tensor cores (bf16 operands, fp32 accumulation), PaTH and PaTH-FoX alike
 * (PaTH-FoX with scale 0 excepted); every other case runs in fp32 on the CUDA
 * cores (bf16 values converted on load and store).  desc->chunk: 16, 32, 64
 * or 128, or 0 for the default of the forward's CUDA-core route; it need not
 * match the chunk the forward used.  Supported: head_dim <= 128 and a
 * multiple of 4.
 * Pointers must be 16-byte aligned.  Argument errors are returned before
 * any launch; the call is asynchronous on `stream`.
 */
path_status_t path_attn_prefill_bwd(const path_prefill_desc_t *desc, const void *q,
                                    const void *k, const void *v, const void *w,
                                    const float *beta, const float *log_f, const void *out,
                                    const float *lse, const void *dout, const float *dlse,
                                    void *dq, void *dk, void *dv, void *dw, float *dbeta,
                                    float *dlog_f, void *workspace, size_t workspace_bytes,
                                    path_stream_t stream);

/* ------------------------------------------------------------------- decode */

typedef struct {
    int32_t batch, heads, head_dim;
    int32_t cache_capacity; /* slots per (batch, head) in the caches */
    int32_t dtype;          /* path_dtype_t; PATH_BF16 only */
    float scale;
} path_decode_desc_t;

/* Bytes of device workspace path_attn_decode_step needs for any cache_len
 * up to the capacity (split-KV partial results); 0 if desc is invalid. */
size_t path_attn_decode_workspace_size(const path_decode_desc_t *desc);

/*
 * One PaTH decode step (section "3. 효율적인 학습 및 추론", inference
 * bullet): every cached key j < cache_len is updated in place with the new
 * token's transition, k_j <- k_j - beta_t w_t (w_t^T k_j), so the cache never
 * stores w; then (k_t, v_t) is written to slot cache_len untransformed and
 *     out = softmax_j(scale * q_t . k_j) v_j   over j <= cache_len.
 *   k_cache, v_cache : [B][H][cache_capacity][d], desc->dtype; k_cache
 *                      slots < cache_len are rewritten, slot cache_len of
 *                      both caches receives k_t / v_t.
 *   q_t, k_t, v_t, w_t : [B][H][d]; beta_t : float32 [B][H]; out : [B][H][d].
 *   cache_len        : tokens already cached, 0 <= cache_len < capacity.
 * The caller advances cache_len by one after the call.  Keys are re-rounded
 * to the cache dtype after every update.
 */
path_status_t path_attn_decode_step(const path_decode_desc_t *desc, void *k_cache,
                                    void *v_cache, int32_t cache_len, const void *q_t,
                                    const void *k_t, const void *v_t, const void *w_t,
                                    const float *beta_t, void *out, void *workspace,
                                    size_t workspace_bytes, path_stream_t stream);

/*
 * One PaTH-FoX decode step: path_attn_decode_step with the forget-gate bias
 * of the PaTH-FoX combination (section "2. 방법론: PaTH Attention", FoX; at
 * inference, section "3. 효율적인 학습 및 추론").  The logit of cached key
 * j < t gains sum_{s=j+1}^{t} log f_s; the new token's own logit gains
 * nothing.  The bias is kept as a prefix per key:
 *   f_cache    float32 [batch, heads, cache_capacity], f_cache[j] =
 *              F_j = sum_{s<=j} log f_s for j < cache_len (read); the step
 *              writes F_t = F_{t-1} + log_f_t at slot cache_len (F_{-1} = 0),
 *              so the bias is F_t - F_j.  After a prefill, fill it with
 *              path_attn_fox_prefix.
 *   log_f_t    float32 [batch, heads]: log of the new token's forget gate.
 * Every other argument, the layouts, ownership, errors and the in-place
 * update are those of path_attn_decode_step.  f_cache and log_f_t need 4-byte
 * alignment.
 */
path_status_t path_attn_decode_step_fox(const path_decode_desc_t *desc, void *k_cache,
                                        void *v_cache, float *f_cache, int32_t cache_len,
                                        const void *q_t, const void *k_t, const void *v_t,
                                        const void *w_t, const float *beta_t,
                                        const float *log_f_t, void *out, void *workspace,
                                        size_t workspace_bytes, path_stream_t stream);

/*
 * Prefix sums of forget-gate logs for the PaTH-FoX decode cache:
 *   f_out[h][i] = sum_{s<=i} log_f[h][s]   for i < len,
 *   f_out[h][i] = f_out[h][len-1]          for len <= i < out_len,
 * summed in fp64, stored as float32.  log_f: [heads_total][len], f_out:
 * [heads_total][out_len] (heads_total = batch * heads), device pointers,
 * caller-owned.  Asynchronous on `stream`.  PATH_ERR_INVALID_ARG for NULL
 * pointers or sizes outside 1 <= len <= out_len, heads_total >= 1.
 */
path_status_t path_attn_fox_prefix(const float *log_f, float *f_out, int32_t heads_total,
                                   int32_t len, int32_t out_len, path_stream_t stream);

/*
 * path_attn_decode_step without a workspace, for callers that cannot
 * allocate device memory: plugins running inside a host framework that owns
 * all GPU memory and gives them no allocator, and token loops that must not
 * call cudaMalloc because it can synchronise the device.  The PaTH pages have
 * no counterpart to this call; it computes exactly what path_attn_decode_step
 * computes, with the same arguments minus the workspace.
 *
 * The split-KV partial results live in one fixed device array of 8 MiB that
 * every GPU loading the library holds until the process exits.  A step needs
 * batch * heads * ceil(cache_len / 1024) * (head_dim + 2) * 4 bytes of it;
 * larger steps are rejected with PATH_ERR_INVALID_ARG and a message naming
 * both sizes (use path_attn_decode_step then).  The first call in each CUDA
 * context looks up the array's device address (cudaGetSymbolAddress) with
 * that context current and caches it for that context (a context made after
 * a device reset gets a fresh lookup); make that first call before any
 * stream capture.  All calls
 * share the one array, which keeps the last call's contents, so calls that
 * overlap on the GPU (different streams, or different host threads on the
 * same device) race with each other: serialise them.  Nothing is allocated
 * or freed by this call.
 */
path_status_t path_attn_decode_step_noalloc(const path_decode_desc_t *desc, void *k_cache,
                                            void *v_cache, int32_t cache_len, const void *q_t,
                                            const void *k_t, const void *v_t, const void *w_t,
                                            const float *beta_t, void *out,
                                            path_stream_t stream);

/*
 * Key cache after a prefill of seq_len tokens, as the decode step expects it:
 *     k_cache[j] = H_{L-1} ... H_{j+1} k_j    (j < L = desc->seq_len),
 * i.e. every key transformed by all later transitions (inference bullet of
 * section 3).  The PaTH pages only describe the in-place update one step at
 * a time; this call produces the same state in O(L d^2) per head by a
 * right-to-left sweep over chunk products.  k, w: [B][H][L][d]; beta:
 * float32 [B][H][L]; k_cache: [B][H][cache_capacity][d] (slots < L written).
 * desc->dtype must equal the cache dtype (PATH_BF16).  The workspace must
 * hold path_attn_build_kcache_workspace_size(desc) bytes.
 */
size_t path_attn_build_kcache_workspace_size(const path_prefill_desc_t *desc);
path_status_t path_attn_build_kcache(const path_prefill_desc_t *desc, const void *k,
                                     const void *w, const float *beta, void *k_cache,
                                     int32_t cache_capacity, void *workspace,
                                     size_t workspace_bytes, path_stream_t stream);

/* ------------------------------------------------- sequence-sharded prefill */

/*
 * The prefill of one long sequence split over `world` ranks, one GPU each
 * (sequence or context parallelism).  The pages' blockwise algorithm
 * (section "3. 효율적인 학습 및 추론", FlashAttention-style algorithm) makes
 * every query chunk scan all earlier key chunks right to left, so the only
 * exchange is the key side of every chunk: its boundary-adjusted keys Kh, its
 * chunk product Pm and its values V, gathered once.
 *
 * Partition.  The N = ceil(seq_len / 128) chunks of 128 positions form
 * 2 * world blocks of nb = ceil(N / (2 * world)) chunks; rank r holds blocks
 * r and 2 * world - 1 - r (a zigzag, so every rank has early and late query
 * chunks and the causal work is balanced).  A rank's local rows are the
 * positions of its two blocks, in order, positions >= seq_len left out;
 * path_attn_cp_local_len gives their number Lr and path_attn_cp_rows lists
 * them.  Local tensors are [batch][heads][Lr][...] in that row order.
 *
 * Per rank:
 *   1. path_attn_cp_prep on the rank's local q, k, v, w, beta: the UT
 *      transform of each local chunk, its boundary-adjusted rows, its chunk
 *      product and its attention to itself; writes the rank's exchange block
 *      (path_attn_cp_exchange_bytes bytes) and keeps the rest in `workspace`.
 *   2. The caller gathers the exchange blocks of all ranks, in rank order,
 *      into one buffer of world * path_attn_cp_exchange_bytes bytes (an
 *      all-gather: ncclAllGather, torch.distributed.all_gather_into_tensor).
 *   3. path_attn_cp_scan with the gathered buffer and the same workspace:
 *      the scan of the rank's query chunks over all earlier chunks; writes
 *      out [batch][heads][Lr][128] and lse [batch][heads][Lr] (or NULL).
 * With world = 1 the two calls compute exactly what path_attn_prefill_fwd
 * computes.  PaTH-FoX: log_f is the forget-gate log of the WHOLE sequence,
 * float32 [batch][heads][seq_len] on every rank (4 bytes per position; the
 * bias needs prefix sums over all earlier positions), given to both calls;
 * NULL for PaTH.  Supported: PATH_BF16, head_dim 128, chunk 0 or 128 (else
 * PATH_ERR_UNSUPPORTED); 1 <= world <= 4096, 0 <= rank < world.  A rank may
 * hold no rows (Lr = 0) when seq_len is short; its calls then read no input,
 * but its exchange block must still take part in the gather.  Pointers are
 * device pointers, 16-byte aligned; calls are asynchronous on `stream`.
 */
int32_t path_attn_cp_local_len(const path_prefill_desc_t *desc, int32_t world, int32_t rank);
/* rows: HOST array of at least Lr entries, filled with the global position of
 * each local row. */
path_status_t path_attn_cp_rows(const path_prefill_desc_t *desc, int32_t world, int32_t rank,
                                int32_t *rows, int32_t capacity);
size_t path_attn_cp_exchange_bytes(const path_prefill_desc_t *desc, int32_t world);
size_t path_attn_cp_workspace_size(const path_prefill_desc_t *desc, int32_t world);
path_status_t path_attn_cp_prep(const path_prefill_desc_t *desc, int32_t world, int32_t rank,
                                const void *q, const void *k, const void *v, const void *w,
                                const float *beta, const float *log_f, void *exchange,
                                void *workspace, size_t workspace_bytes, path_stream_t stream);
path_status_t path_attn_cp_scan(const path_prefill_desc_t *desc, int32_t world, int32_t rank,
                                const float *log_f, const void *exchange_all, void *out,
                                float *lse, void *workspace, size_t workspace_bytes,
                                path_stream_t stream);

/* -------------------------------------------------------------- diagnostics */

/*
 * Synchronises the current device, then reports the device error flag that
 * kernels set when a bounded wait (mbarrier or flag) runs out: PATH_OK,
 * PATH_ERR_TIMEOUT, or PATH_ERR_CUDA if the synchronisation itself failed.
 * clear != 0 resets the flag.
 */
path_status_t path_attn_device_status(int32_t clear);

/*
 * Launches one tiny kernel whose two waits can never complete: one on an
 * mbarrier, one on a global counter (the form in which the scan of
 * path_attn_prefill_fwd waits for the prep's chunks).  Each is bounded by
 * limit_us microseconds of device time; the kernel then sets the device
 * error flag and exits cleanly.  Exists so tests can check the bounded-wait
 * path without hanging a GPU.
 */
path_status_t path_attn_selftest_bounded_wait(uint32_t limit_us, path_stream_t stream);

/* Static text for a status code. */
const char *path_attn_status_string(path_status_t status);

/* Detail message of the last failing call on this host thread ("" if none). */
const char *path_attn_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t path_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PATH_ATTN_H */

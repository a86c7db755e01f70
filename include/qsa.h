/*
 * qsa.h - C ABI of the GB300 (sm_103a) QSA indexer library, libqsa.so.
 *
 * The operation ("spec(MODEL-MM-QWEN4-EXP) ...", section "The component
 * deep-dives", and "[Perf][Qwen4Exp] Admit the cuBLAS QSA indexer and exact
 * top-k on Turing", section "Purpose"):
 *
 *   for every query row r of request b = row_req[r], with V_r = row_visible[r]
 *   visible compressed positions (compress ratio 4, so a query at token t sees
 *   (t+1) // 4 of them):
 *     logit[r, j] = sum_{h<H} w[r,h] * max(q[r,h,:] . k_j, 0)          j < V_r
 *     k_j         = k_cache[block_table[b, j / P], j % P, :]            (paged)
 *   with FP16 q and k, FP32 accumulation; then the exact top-k of row r,
 *   ordered by score descending and, on equal scores, by position ascending
 *   (the "exact lexicographic top-k" with its deterministic tie rule).
 *
 * Conventions shared by every entry point:
 *  - All array arguments are DEVICE pointers into memory the caller owns and
 *    keeps alive until the work on `stream` has finished.  The library never
 *    allocates device memory per call; scratch comes from the caller's
 *    workspace, sized by qsa_workspace_bytes().
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Every call is asynchronous on that stream.
 *  - Host-side argument checks run before any launch and return a status;
 *    nothing is launched when a check fails.  No C++ exception crosses the ABI.
 *    Every int32 / FP32 array must be 4-byte aligned (QSA_ERR_INVALID_ARG
 *    otherwise); stricter alignments are stated where they apply.
 *  - Errors found on the device (bad page id, row_req out of range, a row
 *    longer than the block table or the logit row, a pipeline wait that ran
 *    out of time) never trap: the kernels record them in a per-device status
 *    word and carry on with safe values.  qsa_get_device_status() reads and
 *    clears that word.
 *  - The library keeps per-device state for the life of the process (the
 *    device address of its status word and of its static scratch buffer,
 *    kernel attributes).  A device reset (cudaDeviceReset) invalidates it: do
 *    not call the library on a device after resetting it.
 *  - Supported shapes of the indexer calls: head_dim == 128, H in {1, 2, 4,
 *    8}, page_positions a power of two in [8, 256], 0 <= k <= QSA_MAX_K.  k may
 *    exceed V_r.  Others return QSA_ERR_UNSUPPORTED.  q and k_cache must be
 *    16-byte aligned.  The producer and the consumer (below) state their own.
 *  - Output of the top-k: out_idx[r, 0:min(k, V_r)] holds positions in
 *    (score desc, position asc) order and -1 after that; out_val (optional,
 *    may be NULL) holds the matching logits and -inf after that.
 */
#ifndef QSA_H
#define QSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QSA_MAX_K 8192

typedef enum {
    QSA_OK = 0,
    QSA_ERR_INVALID_ARG = 1,   /* a host-side argument check failed, or (device) row data out of range */
    QSA_ERR_UNSUPPORTED = 2,   /* shape outside the supported set above */
    QSA_ERR_WORKSPACE = 3,     /* workspace NULL or smaller than qsa_workspace_bytes() */
    QSA_ERR_LAUNCH = 4,        /* a kernel launch was refused by the runtime */
    QSA_ERR_BAD_PAGE = 5,      /* (device) a block-table entry outside [0, num_pages) */
    QSA_ERR_TIMEOUT = 6,       /* (device) a pipeline wait ran past its time limit */
    QSA_ERR_CUDA = 7,          /* another CUDA runtime error */
    QSA_ERR_NO_DEVICE = 8,     /* no usable device: the kernels are built for compute capability 10.3 only */
    QSA_ERR_STATIC_LIMIT = 9   /* the call needs more scratch than QSA_STATIC_SCRATCH_BYTES */
} qsa_status;

/* Paged index-key side cache: one FP16 key of head_dim values per compressed
 * position ("a side cache of one index-key vector per token", key only). */
typedef struct {
    const void    *k_cache;            /* device FP16 [num_pages, page_positions, head_dim], contiguous */
    int32_t        num_pages;          /* physical pages in k_cache */
    int32_t        page_positions;     /* positions per page (16 = 64 tokens at ratio 4) */
    int32_t        head_dim;           /* must be 128 */
    const int32_t *block_table;        /* device int32 [num_reqs, max_pages_per_req]: physical page ids */
    int32_t        num_reqs;
    int32_t        max_pages_per_req;  /* row stride of block_table; V_r <= max_pages_per_req * page_positions */
} qsa_paged_keys;

/* Bytes of device workspace the calls below need for `rows` query rows, a
 * top-k of `k` and rows of up to `row_capacity` positions.  row_capacity is
 * the longest row the block table can address, max_pages_per_req *
 * page_positions, NOT the longest visible length of the batch: the workspace
 * is laid out by the block table's capacity.  qsa_index_score needs the size
 * for (rows, 1, 1); qsa_topk_exact needs none.  `flags` is reserved (pass 0).
 * Host only; no device is touched. */
size_t qsa_workspace_bytes(int32_t rows, int32_t row_capacity, int32_t k, int32_t flags);

/* Index scores only: logits[r * ld_logits + j] for 0 <= j < ld_logits, FP32,
 * row-major; -inf for j >= V_r.  q: FP16 [rows, H, 128]; w: FP32 [rows, H];
 * row_req, row_visible: int32 [rows].  Needs ld_logits >= max V_r; a row with
 * V_r > ld_logits is clamped and flagged.  ws/ws_bytes as for the other calls. */
qsa_status qsa_index_score(const void *q, const float *w, int32_t rows, int32_t H,
                           const qsa_paged_keys *keys, const int32_t *row_req,
                           const int32_t *row_visible, float *logits, int64_t ld_logits,
                           void *ws, size_t ws_bytes, void *stream);

/* Exact top-k of each row of a logit matrix (row r holds V_r = row_visible[r]
 * valid entries; entries past V_r are never read).  out_idx: int32 [rows, k];
 * out_val: FP32 [rows, k] or NULL.  Scores must be finite.  ws may be NULL. */
qsa_status qsa_topk_exact(const float *logits, int64_t ld_logits, int32_t rows,
                          const int32_t *row_visible, int32_t k, int32_t *out_idx,
                          float *out_val, void *ws, size_t ws_bytes, void *stream);

/* The whole step: score every visible position of every row, then its exact
 * top-k, without the caller seeing the logits (the operation at the top of
 * this file).  q, w, keys, row_req, row_visible as for qsa_index_score; k,
 * out_idx, out_val as for qsa_topk_exact; ws must hold qsa_workspace_bytes(rows,
 * max_pages_per_req * page_positions, k, 0) bytes, 256-byte aligned.
 * For long rows (at least 3k positions, k >= 342) it scores every 16th key
 * tile (32nd for k >= 2,731) first, takes from that sample a per-row
 * threshold expected to keep 1.5 k positions or more (more for smaller k, so
 * that the expected count stays 4.5 standard deviations above k), scores
 * every tile keeping only the positions at or above it, and
 * selects among those; a row that kept fewer than min(k, V_r) (or too many to
 * hold) is re-scored in plain FP32 and selected from all its positions, so the
 * result never depends on the sample.  Shorter rows are scored into the
 * workspace and selected directly. */
qsa_status qsa_select_paged_tokens(const void *q, const float *w, int32_t rows, int32_t H,
                                   const qsa_paged_keys *keys, const int32_t *row_req,
                                   const int32_t *row_visible, int32_t k, int32_t *out_idx,
                                   float *out_val, void *ws, size_t ws_bytes, void *stream);

/* Synchronises `stream`, then returns and clears the device status word of the
 * current device (QSA_OK when no kernel recorded an error). */
qsa_status qsa_get_device_status(void *stream);

/* ---- Index-key producer: the step before the indexer ----------------------
 * ("spec(MODEL-MM-QWEN4-EXP) ...", section "The component deep-dives": one
 * stored index-key state per four tokens, emitted at the token with
 * (position + 1) % 4 == 0, RMSNorm on the pooled key, RoPE at the block-start
 * position; the DSv4 compress kernel pools with a learned softmax over an
 * overlapping window of eight tokens.)  The pages fix neither the pooling
 * weights nor the RoPE layout; this library's reading:
 *   key_i = RoPE_{4i}( RMSNorm( sum_t a_t * x_t ) )  over the window's tokens t,
 *   a = softmax(pool_logit over the window), or equal weights (the mean) when
 *   pool_logit is NULL; window 4 (the block) or 8 (the block and the four
 *   tokens before it), clipped at position 0; RMSNorm(v) = v / sqrt(mean(v^2)
 *   + eps) * norm_weight; RoPE rotates the pairs (j, j + rope_dim/2),
 *   j < rope_dim/2, by 4i * theta^(-2j/rope_dim) and passes dims >= rope_dim;
 *   the key is rounded to FP16 and stored in keys->k_cache at page
 *   block_table[b][i / P], slot i % P (the cache is written through the
 *   k_cache pointer, which must point to writable device memory).
 *
 * qsa_rope_table: fills table[i * rope_dim + j] = cos(4i * theta^(-2j/rope_dim))
 * and table[i * rope_dim + rope_dim/2 + j] = the sine, for i < n_blocks and
 * j < rope_dim/2, angles in FP64, stored as FP32.  Built once per model; the
 * producer reads row i for block i.  table: device, 16-byte aligned, n_blocks
 * * rope_dim floats.  rope_dim a multiple of 8 in [0, 128]; theta > 0. */
qsa_status qsa_rope_table(float *table, int32_t n_blocks, int32_t rope_dim, double theta, void *stream);

/* qsa_index_key_produce: request b's new tokens are rows seq_start[b] ..
 * seq_start[b+1]-1 of x (FP16 [T, 128], 8-byte aligned), at positions
 * pos_start[b] ..; pool_logit: FP32 [T] or NULL.  Block i of request b is
 * produced when it is complete among the new tokens and every position of its
 * window (from max(0, 4i + 4 - window)) is among them: a decode step that
 * completes a block passes that block's (window's) tokens.  max_tokens: an
 * upper bound of seq_start[b+1] - seq_start[b] (host value; a request with
 * more is flagged and its extra blocks are skipped).  norm_weight: FP32 [128],
 * 16-byte aligned.  rope_table: rope_blocks rows from qsa_rope_table (unused,
 * may be NULL, when rope_dim is 0).  window: 4 or 8 (else
 * QSA_ERR_UNSUPPORTED).  n_reqs <= keys->num_reqs and <= 65535.  Device-side
 * problems (a negative position, a block past the block table or the rope
 * table, a page id outside the cache) skip that block and are reported by
 * qsa_get_device_status(). */
qsa_status qsa_index_key_produce(const void *x, const float *pool_logit, int32_t n_reqs,
                                 const int32_t *seq_start, const int32_t *pos_start, int32_t max_tokens,
                                 const float *norm_weight, float eps, const float *rope_table,
                                 int32_t rope_blocks, int32_t rope_dim, int32_t window,
                                 const qsa_paged_keys *keys, void *stream);

/* ---- Sparse-attention consumer: the step after the indexer ----------------
 * ("spec(MODEL-MM-QWEN4-EXP) ...", section "The component deep-dives": QSA
 * attends raw tokens selected at ratio-4 granularity; plain GQA, 24 query
 * heads over 2 KV heads, head_dim 256.)  This library's reading: row r, a
 * query at token t of request b = row_req[r], attends the tokens 4j .. 4j+3 of
 * every selected index position j = sel[r, 0..k) (as qsa_select_paged_tokens
 * returns them: distinct, below V = (t+1)/4, -1 for none) and the tokens
 * 4V .. t of its unfinished block; query head h reads KV head h / (hq / hkv);
 *   out[r, h, :] = sum_s softmax_s(scale * q[r,h,:] . K[s]) * V[s]
 * q: FP16 [rows, hq, 256]; k_cache, v_cache: FP16 [num_pages, page_tokens,
 * hkv, 256], token p of request b at page block_table[b * max_pages + p /
 * page_tokens], slot p % page_tokens; out: FP32 [rows, hq, 256]; q, the caches
 * and out 16-byte aligned.  head_dim must be 256, hq / hkv <= 16, page_tokens a
 * power of two in [8, 256].  Device-side problems (row_req out of range, a
 * token past the block table, a selected position at or past V, a page id
 * outside the cache) skip the token or the row and are reported by
 * qsa_get_device_status(). */
qsa_status qsa_sparse_attention(const void *q, int32_t rows, int32_t hq, const void *k_cache, const void *v_cache,
                                int32_t num_pages, int32_t page_tokens, int32_t hkv, int32_t head_dim,
                                const int32_t *block_table, int32_t num_reqs, int32_t max_pages,
                                const int32_t *row_req, const int32_t *row_token, const int32_t *sel, int32_t k,
                                float scale, float *out, void *stream);

/* ---- Second workload: the MiniMax-M3-style block scorer ------------------
 * ("spec(MODEL-MM-QWEN4-EXP) ...", section "The component deep-dives", where
 * M3 is set against QSA: a block's score is the maximum of the raw-token
 * query-key dot products over the block, with no pooling, no ReLU and no
 * reduction over heads; index heads equal KV heads, so each query token gets
 * one block set per head; blocks of 128 tokens, the KV page size.)  This
 * library's reading: row r is a query at token t = row_token[r] of request b
 * = row_req[r]; for each head h,
 *   score[r, h, c] = max over tokens p of block c with p <= t of q[r,h,:] . K[p,h,:]
 *   (FP16 inputs, FP32 accumulation), block c holding tokens 128c .. 128c+127,
 * for the blocks c <= t / 128 that hold a visible token; out_idx[r, h, :]
 * holds the top-k blocks by (score desc, block index asc), -1 after them, and
 * out_val (optional) their scores, -inf after them.
 * q: FP16 [rows, H, 128]; k_cache: FP16 [num_pages, 128, H, 128] (one page
 * per block), block c of request b at page block_table[b * max_blocks + c];
 * out_idx int32 / out_val FP32 [rows, H, k].  q and k_cache 16-byte aligned;
 * 1 <= H <= 16; 0 <= k <= QSA_MAX_K.  ws: qsa_block_select_workspace_bytes(rows,
 * H, max_blocks, k) bytes, 256-byte aligned.  Device-side problems (row_req
 * out of range, a negative token, a page id outside the cache) are reported
 * by qsa_get_device_status() (a bad page reads as zeros). */
size_t qsa_block_select_workspace_bytes(int32_t rows, int32_t H, int32_t max_blocks, int32_t k);
qsa_status qsa_block_select(const void *q, int32_t rows, int32_t H, const void *k_cache, int32_t num_pages,
                            const int32_t *block_table, int32_t num_reqs, int32_t max_blocks,
                            const int32_t *row_req, const int32_t *row_token, int32_t k, int32_t *out_idx,
                            float *out_val, void *ws, size_t ws_bytes, void *stream);

/* Static, NUL-terminated description of a status code. */
const char *qsa_status_string(qsa_status status);

/* Tuning / test switches, process-wide (not thread-safe against concurrent
 * calls).  QSA_CFG_PATH: 0 = automatic, 1 = materialise logits then select,
 * 2 = sampled-threshold filter path.  QSA_CFG_WAIT_LIMIT_NS: time after which
 * a pipeline wait gives up and records QSA_ERR_TIMEOUT (default 2 s).
 * Returns QSA_ERR_INVALID_ARG for an unknown key or value. */
#define QSA_CFG_PATH 1
#define QSA_CFG_WAIT_LIMIT_NS 2
#define QSA_CFG_KERNEL_TIMING 3   /* 1: bracket every launch with CUDA events on its stream */
/* 1 (default): the second and later kernels of a call are launched with
 * programmatic stream serialization, so each is scheduled while its
 * predecessor finishes and waits for it on the device before touching memory;
 * 0: plain stream order.  The first kernel of a call always waits for all of
 * the caller's earlier work on the stream. */
#define QSA_CFG_OVERLAP 4
/* CTAs per row of the exact candidate selector on the filter path.  2, 4 or
 * 8: each row goes to one thread-block cluster of that size, whose CTAs
 * gather, count and order slices of the row and merge them through
 * distributed shared memory; the size is capped by what the device's
 * occupancy query (cudaOccupancyMaxPotentialClusterSize) reports it can
 * co-schedule, and a refused launch is retried at half the size down to one
 * CTA per row.  0 (default, automatic) and 1: one CTA per row, which measured
 * faster on every batch tried (on the 64-row decode batch, 18.1 us against
 * 18.6 / 24.4 / 58.6 us for clusters of 2 / 4 / 8).  ("qwen4_exp QSA
 * cooperative_topk cannot launch on NVIDIA Thor (sm_110)": a cluster size
 * must come from the device, not from its compute capability.) */
#define QSA_CFG_CLUSTER 5
qsa_status qsa_set_config(int32_t key, int64_t value);

/* CTAs per row (cluster size) of the most recent launch of the candidate
 * selector in this process; 1 when it ran one CTA per row. */
int32_t qsa_last_cluster_size(void);

/* Kernel kinds reported by qsa_kernel_times(). */
#define QSA_KERNEL_KINDS 10
/* 0 plan, 1 score (logits), 2 score (sampled tiles), 3 score (threshold filter),
 * 4 score (block maxima, qsa_block_select), 5 select (dense rows), 6 select
 * (threshold), 7 select (candidates, including rows re-scored in place),
 * 8 reserved (not launched), 9 -inf padding. */

/* With QSA_CFG_KERNEL_TIMING on: synchronises the pending events, adds each
 * launch's elapsed time to ms[kind] and its count to launches[kind] for the
 * first n kinds (either array may be NULL), then forgets the events.
 * Returns QSA_ERR_CUDA if an event could not be read. */
qsa_status qsa_kernel_times(double *ms, int32_t *launches, int32_t n);

/* Launches made by the most recent qsa_* call on this host thread (kernels of
 * this library only). */
int32_t qsa_last_launch_count(void);

/* qsa_select_paged_tokens for callers that cannot allocate device memory.
 * (This entry point has no counterpart in the pages; it is a convenience of
 * this library.)  Some callers have no device allocator on their hot path:
 * runtimes whose whole device memory is planned once at start-up (a fixed
 * arena, an embedded or safety-certified deployment) must not call
 * cudaMalloc, and may have nowhere to keep a caller-owned workspace either.
 * This variant takes the same arguments minus the workspace and uses a
 * scratch buffer of QSA_STATIC_SCRATCH_BYTES that lives in the library itself
 * (a file-scope __device__ array, present on every GPU that loads the library
 * until the process exits).  It calls no allocating routine.
 *  - The first call on a device looks up that buffer's device address for the
 *    current device; make that first call before any stream capture.
 *  - Calls whose workspace (qsa_workspace_bytes for the same rows, k and
 *    max_pages_per_req * page_positions) exceeds QSA_STATIC_SCRATCH_BYTES
 *    return QSA_ERR_STATIC_LIMIT and launch nothing.
 *  - Every call on a device shares the one buffer and it keeps the previous
 *    call's contents; nothing in it needs to start at zero (each call writes
 *    every region before reading it).  Calls that overlap on the GPU (other
 *    streams, other host threads) race on the buffer: serialise them. */
#define QSA_STATIC_SCRATCH_BYTES (64u << 20)
qsa_status qsa_select_paged_tokens_noalloc(const void *q, const float *w, int32_t rows, int32_t H,
                                           const qsa_paged_keys *keys, const int32_t *row_req,
                                           const int32_t *row_visible, int32_t k, int32_t *out_idx,
                                           float *out_val, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* QSA_H */

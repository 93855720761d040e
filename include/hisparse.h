/*
 * hisparse.h -- C ABI of the Hybrid HiSparse decode hot path on GB300 (sm_103a).
 *
 * One decode step of sparse-MLA attention with KV offloading, as described by
 * "vLLM introduces Hybrid HiSparse hybrid sparse offloading for GLM 5.3"
 * (vLLM blog Part 1; cited below as [P1]) and "Serving GLM-5.3 with PCP, DCP and
 * Hybrid HiSparse" (vLLM blog Part 2; [P2]):
 *
 *   hs_append_rows        write the step's new KV rows and index keys
 *   hs_indexer_topk       score every earlier token, keep the top K    [P2 "Why not TP or DP?"]
 *   hs_resolve_topk       map each selected token to a KV row id       [P1 "How it works"]
 *   hs_replay_topk        the same row ids again, without touching the LRU state
 *                         (verification reruns)                         [P1 "Composing with the rest of vLLM"]
 *   hs_sparse_mla_decode  attention over only those rows               [P2 footnote 1]
 *   hs_offload_pages      copy completed pages of all layers to host   [P1 "How it works"]
 *
 * Conventions
 * - Every call returns an hs_status. No C++ exception crosses the ABI.
 * - Every call opens an NVTX range named after it (inert unless a profiler is
 *   attached), so a timeline shows the decode step call by call.
 * - "d_" pointers are device memory, "h_" pointers are host memory. The big
 *   buffers (KV pool tensors, index-key caches, pinned host pool) are owned by
 *   the caller and must outlive the pool. The library owns only the opaque
 *   hs_pool and its device metadata, allocated by hs_pool_init and freed by
 *   hs_pool_destroy. No call between hs_pool_init and hs_pool_destroy
 *   allocates device memory or page-locked host memory (the first launch of each
 *   kernel on a device only records its attributes in a small host-side table).
 * - Hot-path calls (hs_append_rows .. hs_offload_pages) are asynchronous on the
 *   given stream, do not synchronise with the host and read no device data on
 *   the host, so a sequence of them can be captured in a CUDA graph. Errors the
 *   kernels detect (bad ids, a miss with no host copy, hot-buffer overflow, a
 *   timed-out wait) are recorded in a device status word and reported by
 *   hs_get_error, which synchronises the stream. A call that finds a bad
 *   argument on the host returns HS_ERR_INVALID and launches nothing.
 * - Programmatic dependent launch: a hot-path kernel may start while the previous
 *   kernel of the stream finishes, and waits for it before it reads the outputs of
 *   earlier calls of this library (scores, top-K, row ids, KV rows and index keys).
 *   A call's own input arrays (d_req, d_limit, d_pos, the rows and keys to append,
 *   the indexer's d_q and d_w, the attention's d_q), the block tables and the
 *   hot-buffer state are read before that wait, so they must be final before the
 *   previous kernel started. That holds for values written by the host (copies are
 *   stream-ordered), by this library's own calls (none writes them in a kernel) and
 *   by any ordinary kernel launch, which lets no dependent start before it ends; it
 *   does not hold for a kernel that itself lets its dependents start early
 *   (griddepcontrol.launch_dependents) and writes them afterwards.
 * - A query-token batch is described by per-token device arrays: d_req (the
 *   request slot of each token) and d_limit (causal limit: the token sees
 *   positions [0, limit)). The tokens of one request are contiguous in the
 *   batch, at most max_q_per_req of them, in ascending position.
 * - bf16 values are passed as uint16_t bit patterns.
 */
#ifndef HISPARSE_H
#define HISPARSE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Longest context a pool accepts (tokens per request). The cluster top-K selection
 * (a middling number of query tokens, and hs_indexer_topk_noalloc) splits a token's
 * scores over a 16-CTA cluster and keeps a 2-byte bucket per score of its share in
 * shared memory, which bounds the share at 81,920 scores. (With few query tokens the
 * selection spreads each token over up to one CTA per SM, holding at most 12,288 scores
 * per CTA; with many it cuts each token into chunks of 8,192 scores.) */
#define HS_MAX_CTX 1310720

typedef struct CUstream_st* hs_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum hs_status {
  HS_OK = 0,
  HS_ERR_INVALID = 1,      /* bad argument found on the host; nothing launched */
  HS_ERR_OOM = 2,          /* hs_pool_init could not allocate its metadata */
  HS_ERR_CAPACITY = 3,     /* device: more misses than evictable hot-buffer slots */
  HS_ERR_CUDA = 4,         /* a CUDA runtime call failed */
  HS_ERR_TIMEOUT = 5,      /* device: a bounded wait inside a kernel gave up */
  HS_ERR_HOST_MISSING = 6, /* device: a placeholder page without a host copy was selected */
  HS_ERR_BAD_ID = 7,       /* device: a page, row or token id out of range */
  HS_ERR_BAD_WEIGHT = 8,   /* device: a negative index-head weight */
  HS_ERR_SCRATCH_LIMIT = 9, /* request larger than the fixed scratch of hs_indexer_topk_noalloc */
  HS_ERR_NOT_RESOLVED = 10, /* hs_replay_topk met a token that is neither resident nor hot */
  HS_ERR_RANGE = 11         /* device: an attention input beyond the fp16 range of the batched path */
} hs_status;

/* Index-key formats.
 * HS_IDX_INT8: 128 int8 values per key; a page of a key cache is [64][128] int8
 *   (8,192 bytes); scores are exact int64 (hs_indexer_topk).
 * HS_IDX_FP8: the pages' key record ([P2] footnote 3: 128 FP8 values plus a 4-byte
 *   scale, 132 bytes): a page is 64 x 128 e4m3 bytes followed by the 64 keys' fp32
 *   scales (8,448 bytes, HS_IDX_FP8_PAGE_BYTES); scores are fp32
 *   (hs_indexer_topk_fp8). */
#define HS_IDX_INT8 0
#define HS_IDX_FP8 1
#define HS_IDX_FP8_PAGE_BYTES 8448

/* Pool geometry. Sizes are fixed for the pool's lifetime. */
typedef struct hs_pool_config {
  int32_t page_size;          /* tokens per page; must be 64 */
  int32_t row_bytes;          /* bytes per KV row; must be 656 ([P2] footnote 1, fp8_ds_mla) */
  int32_t idx_dim;            /* index key dims; must be 128 */
  int32_t n_idx_heads;        /* H_i: 16, 32, 48 or 64 */
  int32_t n_heads;            /* attention heads H: 16, 32 or 64 */
  int32_t topk;               /* K: multiple of 128, 128..2048 */
  int32_t n_layers;           /* sparse-MLA layers, 1..64 */
  int32_t layers_per_indexer; /* IndexShare group size ([P1] "Sparsity when you need it"), 1..8 */
  int32_t num_pages;          /* pool pages in each layer's KV tensor, >= 1, num_pages * 64 < 2^31 */
  int32_t num_idx_pages;      /* pages in each indexer layer's key cache, >= 1 */
  int32_t max_requests;       /* request slots */
  int32_t max_ctx;            /* max positions per request, multiple of 128, <= HS_MAX_CTX */
  int32_t max_q_per_req;      /* query tokens per request per call, 1..4 */
  int32_t hot_rows;           /* hot-buffer capacity per (request, group), multiple of 64, 64..16384 */
  int32_t max_tokens;         /* query tokens per call, 1..1024 */
  int32_t idx_format;         /* index-key format: HS_IDX_INT8 or HS_IDX_FP8 */
  int64_t host_pages;         /* pages in the pinned host pool, >= 1 */
} hs_pool_config;

/* One resolved selection ([P1] "How it works": resident / hot / miss). */
typedef struct hs_plan_entry {
  int32_t kind;    /* 0 pad (-1 in top-K), 1 resident, 2 hot-buffer hit, 3 miss */
  int32_t slot;    /* hot-buffer slot for hit and miss, else -1 */
  int32_t row;     /* HMA row id = pool page * 64 + offset, -1 for pad */
  int32_t evicted; /* token whose slot a miss took over, else -1 */
} hs_plan_entry;

/* Running counters kept on the device, read by hs_get_counters. */
typedef struct hs_counters {
  uint64_t resident;   /* distinct selected tokens read in place */
  uint64_t hits;       /* distinct selected tokens found in the hot buffer */
  uint64_t misses;     /* distinct selected tokens copied from host */
  uint64_t h2d_bytes;  /* bytes copied host -> device by misses (656 per row per layer) */
  uint64_t d2h_bytes;  /* bytes copied device -> host by hs_offload_pages */
  uint64_t reserved[3];
} hs_counters;

typedef struct hs_pool hs_pool;

/* Check a pool geometry without touching the GPU: HS_OK if hs_pool_init would
 * accept it (the limits listed in hs_pool_config), HS_ERR_INVALID otherwise (or
 * for a NULL cfg). hs_pool_init applies the same check first. */
hs_status hs_pool_config_check(const hs_pool_config* cfg);

/*
 * Create a pool over caller-owned memory.
 *  cfg         geometry (copied).
 *  d_kv_layers n_layers device pointers, each [num_pages, 64, 656] bytes, 16-byte aligned.
 *              Row layout: 512 FP8 e4m3 latent, 4 fp32 scales (one per 128 latent
 *              values), 64 bf16 rope values, little endian.
 *  d_idx_layers ceil(n_layers / layers_per_indexer) device pointers, each a key
 *              cache of num_idx_pages pages in cfg.idx_format's page layout
 *              (HS_IDX_INT8: [64][128] int8; HS_IDX_FP8: [64][128] e4m3 then [64]
 *              fp32 scales), 16-byte aligned.
 *  h_host_kv   pinned, mapped host memory of host_pages * n_layers * 64 * 656 bytes,
 *              layout [host_page][layer][64][656] (cudaHostAlloc or torch pin_memory).
 *  out         receives the pool.
 * Allocates the per-request metadata (block tables, hot-buffer state, scratch)
 * on the current device and initialises it: every page a placeholder, every hot
 * buffer empty. Errors: HS_ERR_INVALID (bad geometry, null or misaligned
 * pointer, host memory not mapped), HS_ERR_OOM, HS_ERR_CUDA.
 */
hs_status hs_pool_init(const hs_pool_config* cfg, void* const* d_kv_layers,
                       void* const* d_idx_layers, void* h_host_kv, hs_pool** out);

/* Synchronises the device and frees everything hs_pool_init allocated. */
hs_status hs_pool_destroy(hs_pool* pool);

/* ---------------------------------------------------------------------------
 * Host-side residency updates, issued between steps (stream-ordered copies of
 * small host arrays, which the call takes by value: the arrays, page-locked or
 * not, may be reused as soon as the call returns; those copies from pageable host
 * memory make hs_request_set_pages and hs_hot_lease not graph-capturable).
 * ------------------------------------------------------------------------- */

/* Set n consecutive logical pages [first_page, first_page + n) of request req.
 *  h_block_table  pool page or -1 (placeholder: the page lives on the host only);
 *                 [P1] "How it works": the block table holds real blocks and
 *                 empty placeholders.
 *  h_idx_pages    index-key cache page of each logical page (always resident).
 *  h_host_pages   host page holding the page's materialised copy, or -1.
 * Any of the three may be NULL to leave that table unchanged. */
hs_status hs_request_set_pages(hs_pool* pool, int32_t req, int32_t first_page, int32_t n,
                               const int32_t* h_block_table, const int32_t* h_idx_pages,
                               const int64_t* h_host_pages, hs_stream_t stream);

/* Lease n more pool pages to the hot buffer of (req, group): their 64 * n slots
 * follow the existing ones. Hot pages are ordinary pool pages from the same KV
 * tensors ([P1] "How it works"). Total leased rows must stay <= hot_rows. */
hs_status hs_hot_lease(hs_pool* pool, int32_t req, int32_t group, int32_t n,
                       const int32_t* h_pool_pages, hs_stream_t stream);

/* Empty every hot buffer of req (request end); the caller takes the pages back. */
hs_status hs_hot_release(hs_pool* pool, int32_t req, hs_stream_t stream);

/* ---------------------------------------------------------------------------
 * Device hot path (graph-capturable).
 * ------------------------------------------------------------------------- */

/* Write the KV row of every sparse layer and the index key of every indexer
 * layer for n_tokens new positions.
 *  d_req, d_pos   [n] request slot and position of each new row.
 *  d_kv_rows      [n, n_layers, 656] bytes; d_idx_keys [n, n_idx_layers, R] bytes,
 *                 R = 128 (HS_IDX_INT8: int8 values) or 132 (HS_IDX_FP8: 128 e4m3
 *                 values then the key's fp32 scale, little endian).
 * The page holding each position must be resident (block table >= 0). */
hs_status hs_append_rows(hs_pool* pool, int32_t n_tokens, const int32_t* d_req,
                         const int32_t* d_pos, const uint8_t* d_kv_rows,
                         const int8_t* d_idx_keys, hs_stream_t stream);

/* Indexer scores and top-K for one indexer layer ([P2] "Why not TP or DP?": the
 * indexer scores every earlier token to pick the 2,048 that sparse MLA attends to).
 *  s[t] = sum_h w[h] * max(0, sum_d q[h][d] * key_t[d]) exact in int64, t < limit.
 *  d_q [n, H_i, 128] int8, d_w [n, H_i] int8 (must be >= 0).
 *  d_topk [n, K] int32 out: the K highest scores, ties to the lower token, in
 *  ascending token order; -1 pads when limit < K.
 *  d_scores nullable [n, max_ctx] int64 out, 16-byte aligned: every score (entries >= limit
 *  undefined).
 * Selection on the whole GPU: with few query tokens the top-K selection spreads each
 * token over up to one CTA per SM and synchronises them with bounded grid-wide
 * waits, which needs every one of those CTAs resident at once. Work on other streams
 * that holds SMs for longer than the one-second wait limit makes the call fail with
 * HS_ERR_TIMEOUT (read by hs_get_error, which also clears the selection scratch the
 * timed-out call left). hs_set_select_mode(pool, HS_SELECT_LOCAL) avoids this path
 * for engines that share the GPU; the no-allocation variant below never uses it.
 * With many query tokens (up to one per SM) each token's scores are cut into chunks
 * spread over the GPU with no cross-CTA waits; beyond that, one CTA per token. The
 * chunked path keeps about 65 KB of scratch per query token of the pool (max_tokens) and,
 * like the wide one, assumes one call at a time per pool. */
hs_status hs_indexer_topk(hs_pool* pool, int32_t index_layer, int32_t n_tokens,
                          const int32_t* d_req, const int32_t* d_limit, const int8_t* d_q,
                          const int8_t* d_w, int32_t* d_topk, int64_t* d_scores,
                          hs_stream_t stream);

/* FP8 indexer and top-K for a pool with idx_format HS_IDX_FP8 ([P2] footnote 3:
 * keys of 128 FP8 values and a 4-byte scale). Per query token j and earlier
 * token t:
 *   s[t] = scale_t * sum_h w[h] * max(0, sum_d q[h][d] * k_t[d])   (fp32)
 * with q and k e4m3; a query's own scale is folded into its head weights w (fp32,
 * any sign). The top K by (s descending, t ascending), ascending, -1 pads.
 *  d_q [n, H_i, 128] e4m3, 16-byte aligned; d_w [n, H_i] fp32; d_topk [n, K] out;
 *  d_scores nullable [n, max_ctx] fp32 out (entries >= limit untouched).
 * HS_ERR_INVALID on a pool of the other format. */
hs_status hs_indexer_topk_fp8(hs_pool* pool, int32_t index_layer, int32_t n_tokens, const int32_t* d_req,
                              const int32_t* d_limit, const uint8_t* d_q, const float* d_w, int32_t* d_topk,
                              float* d_scores, hs_stream_t stream);

/* Fused top-K resolver for indexer group `group` at step `step` ([P1] "How it
 * works"): for the union of the selected tokens of each request, a resident page
 * is read in place, a hot-buffer hit refreshes its LRU stamp, and a miss takes
 * the least recently used slot (stamp, then slot, ascending; empty slots first)
 * and copies that token's row of every layer of the group from the pinned host
 * pool into it. step must increase from call to call for a given (req, group).
 *  d_topk [n, K] as hs_indexer_topk writes it: each row ascending, -1 pads at
 *  the end (ids >= max_ctx set HS_ERR_BAD_ID and count as pads); d_row_ids [n, K]
 *  out (-1 for pads);
 *  d_plan nullable [n, K] out. */
hs_status hs_resolve_topk(hs_pool* pool, int32_t group, int32_t step, int32_t n_tokens,
                          const int32_t* d_req, const int32_t* d_topk, int32_t* d_row_ids,
                          hs_plan_entry* d_plan, hs_stream_t stream);

/* Replay of a resolver plan for a verification rerun ([P1] "Composing with the
 * rest of vLLM": speculative decoding works through per-step replayable resolver
 * plans that share the request's hot state). Maps each selected token to the row
 * the last hs_resolve_topk of group `group` gave it, from the residency maps as
 * they stand, and changes nothing: no LRU stamp is refreshed, no slot is taken, no
 * row is copied, no counter moves. Every selected token must be resident or hold a
 * hot slot (as right after hs_resolve_topk of the same selection); one that holds
 * neither gets row id -1 and sets HS_ERR_NOT_RESOLVED in the device status word.
 *  d_req [n], d_topk [n, K] as for hs_resolve_topk; d_row_ids [n, K] out (-1 for
 *  pads). Graph-capturable; one launch. */
hs_status hs_replay_topk(hs_pool* pool, int32_t group, int32_t n_tokens, const int32_t* d_req,
                         const int32_t* d_topk, int32_t* d_row_ids, hs_stream_t stream);

/* Sparse MLA decode for one layer ([P2] footnote 1; MQA form: every row serves
 * all heads). Per token and head: z_t = sm_scale * q . k_t over the 576 dims
 * (512 dequantised latent + 64 rope) of each selected row, o = softmax(z) . v_t
 * over the 512 latent dims, lse = log sum exp z.
 *  d_q [n, H, 576] bf16, 16-byte aligned; d_row_ids [n, K] (-1 skipped);
 *  d_out [n, H, 512] bf16, 16-byte aligned; d_lse nullable [n, H] fp32. d_out
 *  may also be pinned, mapped host memory (the kernel then writes the output over
 *  the host link itself, with no copy afterwards).
 *  Per-group FP8 scales must be below 256 (HS_ERR_INVALID for misaligned
 *  pointers or out-of-range arguments).
 *  Layers of one selection: when the previous launch of this pool was
 *  hs_sparse_mla_decode with the same d_row_ids on the same stream, the kernel
 *  also reads the row ids and gathers the rows while that kernel finishes
 *  (programmatic dependent launch).
 *  Between two such calls, d_row_ids and the KV rows may change only through
 *  stream work that is not a programmatic-dependent kernel (an ordinary kernel
 *  launch, a copy or a memset). Any other call of this library on the pool ends
 *  the pairing. */
hs_status hs_sparse_mla_decode(hs_pool* pool, int32_t layer, int32_t n_tokens,
                               const uint16_t* d_q, const int32_t* d_row_ids, float sm_scale,
                               uint16_t* d_out, float* d_lse, hs_stream_t stream);

/* Copy n pool pages of every sparse layer to their host pages in one launch
 * ([P1] "How it works": all sparse-MLA layers are copied in one launch after the
 * forward pass, ordered on the model's stream).
 *  d_pool_pages [n] int32, d_host_pages [n] int64. */
hs_status hs_offload_pages(hs_pool* pool, int32_t n, const int32_t* d_pool_pages,
                           const int64_t* d_host_pages, hs_stream_t stream);

/* hs_indexer_topk for callers that cannot allocate device memory. The pages have
 * no counterpart; this is a deployment variant of the call above.
 * Who needs it: an engine that gives all free HBM to its KV pool before serving
 * (a later cudaMalloc fails or fragments the pool), or code running while a
 * stream is captured, where cudaMalloc is not allowed.
 * What differs: the int64 score scratch is a fixed array inside the library,
 * HS_NOALLOC_MAX_SCORES entries (16 MiB), held by every GPU that loads the
 * library until the process exits; the call allocates nothing and uses no
 * pool-owned scratch. Arguments and results are those of hs_indexer_topk
 * without d_scores.
 * Limits and rules:
 *  - n_tokens * cfg.max_ctx must not exceed HS_NOALLOC_MAX_SCORES, otherwise the
 *    call returns HS_ERR_SCRATCH_LIMIT and launches nothing;
 *  - the pool's device must be current (HS_ERR_INVALID otherwise);
 *  - the first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) and caches it; make that first call before any
 *    stream capture;
 *  - every call on a device shares the one array, which keeps the previous
 *    call's scores (each call writes every score it later reads, nothing needs
 *    clearing); calls whose kernels overlap on the GPU, e.g. on two streams,
 *    race on it and must be ordered by the caller. */
#define HS_NOALLOC_MAX_SCORES (1ll << 21)
hs_status hs_indexer_topk_noalloc(hs_pool* pool, int32_t index_layer, int32_t n_tokens,
                                  const int32_t* d_req, const int32_t* d_limit, const int8_t* d_q,
                                  const int8_t* d_w, int32_t* d_topk, hs_stream_t stream);

/* Self-test of the failure path (not part of the decode step): one kernel waits,
 * with the bounded wait every hot-path kernel uses, for an mbarrier arrival that
 * never comes; after about one second it records HS_ERR_TIMEOUT in the device
 * status word and returns, leaving the context usable. Asynchronous. */
hs_status hs_wait_selftest(hs_pool* pool, hs_stream_t stream);

/* Self-test of the selection's failure path (not part of the decode step). Runs the
 * grid-wide top-K selection again over the scores the pool's last hs_indexer_topk
 * (or hs_indexer_topk_fp8) call left in its scratch (a call made with d_scores
 * NULL), with one CTA of each query token never arriving at the grid-wide waits, as
 * when work on another stream holds an SM. The token's other CTAs give up after
 * about one second: HS_ERR_TIMEOUT in the device status word and a half-used
 * selection scratch, which later selections route around (correct, slower) until
 * hs_get_error reports the timeout and clears it. d_limit [n] as for the indexer;
 * d_topk [n, K] receives undefined values. HS_ERR_INVALID when n tokens would not
 * take the grid-wide selection. Asynchronous. */
hs_status hs_select_selftest(hs_pool* pool, int32_t n_tokens, const int32_t* d_limit, int32_t* d_topk,
                             hs_stream_t stream);

/* Synchronise stream, return the first device-detected error since the last
 * call in *device_status and clear it. When it is HS_ERR_TIMEOUT, the selection
 * scratch a timed-out grid-wide wait may have left half used is also cleared, so
 * later calls run at full speed again (until then they select correctly on a
 * slower path that uses no scratch). The pool's calls must be issued on one
 * stream at a time. */
hs_status hs_get_error(hs_pool* pool, hs_status* device_status, hs_stream_t stream);

/* Selection modes (hs_set_select_mode).
 * HS_SELECT_AUTO   (default) few query tokens are selected by groups of CTAs spread
 *                  over every SM with bounded grid-wide waits (fastest when the
 *                  pool's calls have the GPU to themselves);
 * HS_SELECT_LOCAL  no selection waits on CTAs of other SMs: one CTA, or one
 *                  cluster of CTAs, per query token. For engines that run other
 *                  work on the GPU at the same time. */
#define HS_SELECT_AUTO 0
#define HS_SELECT_LOCAL 1
/* Host-side, between steps. HS_ERR_INVALID for an unknown mode. */
hs_status hs_set_select_mode(hs_pool* pool, int32_t mode);

/* Synchronise stream and read the device counters (reset = nonzero clears them). */
hs_status hs_get_counters(hs_pool* pool, hs_counters* out, int32_t reset, hs_stream_t stream);

/* Static text for a status code. */
const char* hs_status_string(hs_status s);

/* Host-link probe (a measurement aid, not part of the decode step and needing no
 * pool): copies n single rows of row_bytes from pinned, mapped host memory into
 * d_dst, row i taken from host row d_src_rows[i], 16 bytes per thread with four
 * loads in flight, the access pattern of the resolver's miss copies. Timing it
 * gives the host-link rate for single-row reads that the step roofline charges
 * miss bytes against ([P1] "How it works": a miss copies one row from pinned host
 * memory).
 *  h_mapped: pinned host memory allocated mapped (cudaHostAllocMapped, or a
 *  PyTorch pinned tensor), n_host_rows rows of row_bytes, 16-byte aligned;
 *  row_bytes a positive multiple of 16; d_src_rows [n] int64, an index outside
 *  [0, n_host_rows) leaves its destination row unchanged; d_dst
 *  [n * row_bytes], 16-byte aligned. HS_ERR_INVALID for a null or misaligned
 *  pointer, a bad size, or host memory that is not mapped. Asynchronous. */
hs_status hs_link_probe(const void* h_mapped, int64_t n_host_rows, int32_t row_bytes, const int64_t* d_src_rows,
                        int64_t n, void* d_dst, hs_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* HISPARSE_H */

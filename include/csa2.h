/*
 * csa2.h -- C ABI of libcsa2.so: CSA2 sparse decode attention on one GB300.
 *
 * The method (DeepSeek V4.1 Flash, as described on the architecture page
 * k-a.in "DeepSeek V4.1 Flash"):
 *   - section "CSA2 with cross-layer reuse", mode table: a Full layer computes
 *     its own main KV / indexer keys and a fresh Top-K; a Reindex layer reuses
 *     them but runs its own indexer query and a fresh Top-K; a Reuse layer
 *     reuses KV, indexer keys and the Top-K indices.  Every mode computes its
 *     own main query and SWA KV.
 *   - bullet "Sparse attention": each query reads its Top-512 main-KV entries
 *     plus a 128-token sliding window (SWA).
 *   - bullet "Hierarchical indexer": later decoder indexers score at most
 *     16,384 candidates whatever the context length (blocks of 8 entries, a
 *     pool of at most 2,048 blocks); page "DeepSeek V4.1 Flash made encoders
 *     cool" (artofsm.art): the hierarchical sparse indexer narrows candidates
 *     to blocks.
 * The pages do not give the indexer formula (they point to "section 4.2.1" of
 * a report that is not among them).  This library computes, for a query with
 * indexer heads q_h and weights w_h, the score of a key k as
 *     s(k) = sum_h w_h * ReLU(q_h . k)          (ReLU optional, see relu)
 * and selects Top-K under the total order (score descending, index ascending).
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is DEVICE memory owned by the caller, row-major
 *     and contiguous, unless stated otherwise.  Arrays read by bulk copies
 *     (keys, main KV, SWA KV, queries) must be 16-byte aligned.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  No entry point allocates or frees memory, and none
 *     synchronises except csa2_read_device_error and
 *     csa2_read_static_device_error.
 *   - Arguments are validated on the host before anything is enqueued; a
 *     negative csa2_status is returned and nothing is launched.  A failed
 *     launch returns CSA2_ERR_CUDA.
 *   - Conditions only the device can see (an index outside the cache, a count
 *     outside its range, a pooled block id outside the valid blocks) are
 *     clamped or skipped by the kernels and recorded in a sticky error word in
 *     the workspace header; kernels never trap.  Read it with
 *     csa2_read_device_error.
 *   - Kernels are launched with programmatic dependent launch.  Some read
 *     the call's own inputs (q, SWA rows, n_swa, k_swa, v_swa) before waiting
 *     for the preceding kernel of the stream, which is safe under ordinary
 *     stream order.  If the kernel enqueued just before a call lets its
 *     dependents start early (griddepcontrol.launch_dependents), it must not
 *     write those inputs after doing so.  The library's own kernels never
 *     write them; csa2_kv_append and csa2_swa_append, which do, never start
 *     their dependents early.
 *   - `ws` is a caller-owned device workspace of at least
 *     csa2_workspace_bytes(shape) bytes, 256-byte aligned, zeroed once with
 *     csa2_workspace_init before first use.  Calls that share a workspace
 *     must be ordered on one stream.  The cache-maintenance calls
 *     (csa2_block_keys, csa2_kv_append, csa2_swa_append) use only the
 *     workspace's error word; they also accept ws = NULL with ws_bytes = 0,
 *     and then record device errors in the header of the library's static
 *     scratch array (see csa2_layer_group_static), where
 *     csa2_read_static_device_error reads them.
 *   - Element type (csa2_shape.dtype): bf16 or fp32, for queries, keys,
 *     values and indexer tensors alike.  Scores, weights, outputs and lse are
 *     fp32; indices and counts are int32.
 */
#ifndef CSA2_H_
#define CSA2_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* csa2_stream_t; /* identical to cudaStream_t */

typedef enum {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = -1,  /* null pointer, bad size, misaligned pointer, illegal mode sequence */
  CSA2_ERR_UNSUPPORTED = -2,  /* valid but not implemented (e.g. dims beyond the generic limits) */
  CSA2_ERR_WORKSPACE = -3,    /* ws too small or misaligned */
  CSA2_ERR_CUDA = -4,         /* a CUDA launch or runtime call failed */
  CSA2_ERR_DEVICE_CHECK = -5, /* returned by csa2_read_device_error: a kernel recorded a bad input */
  CSA2_ERR_TIMEOUT = -6       /* returned by csa2_read_device_error: a bounded device wait gave up */
} csa2_status;

/* CSA2_SWA: a pure sliding-window layer (the first two encoder layers of the
 * architecture figure caption): it attends only its own SWA rows and neither
 * needs nor produces indices. */
typedef enum { CSA2_FULL = 0, CSA2_REINDEX = 1, CSA2_REUSE = 2, CSA2_SWA = 3 } csa2_mode;
typedef enum { CSA2_BF16 = 0, CSA2_F32 = 1 } csa2_dtype;

/* Problem shape shared by a layer group.  Symbols: B batch (one decode query
 * per sequence), N compressed main-KV entries per sequence (cache capacity),
 * HI x dI indexer heads x dim, P pool blocks, K Top-K, H query heads sharing
 * one KV head with key dim dk and value dim dv, W SWA rows. */
typedef struct {
  int32_t batch;       /* B >= 1 */
  int32_t n_entries;   /* N >= 1; a multiple of `block` when a hierarchical stage is used */
  int32_t idx_heads;   /* HI, 1..64 */
  int32_t idx_dim;     /* dI, 1..1024 */
  int32_t block;       /* entries per block, >= 1 (8 in the architecture) */
  int32_t pool_blocks; /* P: blocks kept by the hierarchical stage; 0 = no hierarchical stage */
  int32_t topk;        /* K, 1..1024 (512 in the architecture) */
  int32_t q_heads;     /* H, 1..1024 */
  int32_t k_dim;       /* dk, 1..1024 */
  int32_t v_dim;       /* dv, 1..1024 */
  int32_t swa;         /* W, 0..1024 (128 in the architecture); K + W <= 1024 */
  float scale;         /* softmax scale; <= 0 selects 1/sqrt(dk) */
  int32_t relu;        /* 1: ReLU on each indexer head's dot product (default reading); 0: none */
  int32_t dtype;       /* csa2_dtype */
  int32_t tokens;      /* T: query tokens per sequence (0 or 1: one).  With T > 1 (architecture
                          page, "Asymmetric encoder-decoder": prompt tokens run a 128-token decoder
                          replay), B is a multiple of T and queries b = s*T .. s*T + T-1 share the
                          caches of sequence s: k_main, v_main and k_idx are then [B / T, N, ...].
                          Everything else stays per query, including n_valid (each token's own
                          causal count), the SWA rows and kb (block summary keys of the query's own
                          valid prefix, so a token's partial last block averages only entries it
                          may see).  csa2_kv_append and csa2_swa_append take T <= 1. */
} csa2_shape;

/* One layer of a group (csa2_layer_group). */
typedef struct {
  int32_t mode;        /* csa2_mode */
  int32_t hier;        /* 1: hierarchical (block pool) indexing; needs kb and pool_blocks > 0 */
  const void* q;       /* [B, H, dk] the layer's own query */
  const void* q_idx;   /* [B, HI, dI] indexer query (Full / Reindex; ignored for Reuse and SWA) */
  const float* w_idx;  /* [B, HI] indexer head weights (Full / Reindex; ignored for Reuse and SWA) */
  const void* k_swa;   /* [B, W, dk] the layer's own SWA keys: rows 0..n_swa-1 in any order
                          (oldest first, or the ring csa2_swa_append keeps) */
  const void* v_swa;   /* [B, W, dv] the layer's own SWA values */
  float* out;          /* [B, H, dv] attention output */
  float* lse;          /* [B, H] natural-log sum of exp of the scaled logits, or NULL */
  int32_t* idx_out;    /* [B, K] fresh indices of an indexing layer, or NULL; untouched for Reuse / SWA */
} csa2_layer;

/* Workspace bytes needed by any entry point for this shape (host only). */
size_t csa2_workspace_bytes(const csa2_shape* shape);

/* Zero the workspace header (device error word).  Call once before first use. */
int csa2_workspace_init(void* ws, size_t ws_bytes, csa2_stream_t stream);

/* Block summary keys (cache-side maintenance, architecture page bullet
 * "Hierarchical indexer"; the 128K Reindex workload defines the summary as
 * the mean of the block's 8 keys rounded to integers).
 * kb[b, j, :] = mean of k_idx[b, j*block + t, :] over the valid entries
 * t < block with j*block + t < n_valid[b] (a partial last block averages its
 * valid entries), rounded half-to-even to an integer if round_to_int, then
 * stored in the element type.  Blocks j >= ceil(n_valid[b] / block) are
 * written as 0.
 *   k_idx   [B, N, dI]     n_valid [B] (0..N)
 *   kb      [B, ceil(N / block), dI]  (output) */
int csa2_block_keys(const csa2_shape* shape, const void* k_idx, const int32_t* n_valid,
                    int32_t round_to_int, void* kb, void* ws, size_t ws_bytes, csa2_stream_t stream);

/* Decode-step cache maintenance, main caches (architecture page: the
 * compressed main KV grows by one entry per compressed span of tokens, and
 * bullet "Hierarchical indexer" keeps one summary key per block of 8 entries;
 * producing the compressed entries themselves is a learned operator the pages
 * do not describe, so they are inputs here).
 * For each query b, the first n_new[b] rows (0..max_new) of k_new[b],
 * v_new[b] and kidx_new[b] are written at entry positions n_valid[b],
 * n_valid[b] + 1, ... of k_main, v_main and k_idx; then, when kb is not NULL,
 * the summary key of every block those positions fall in is recomputed over
 * the block's valid entries exactly as csa2_block_keys computes it (other
 * blocks are left as they are); finally n_valid[b] grows by n_new[b].
 * Entries that would land at N or beyond are dropped and recorded in the
 * device error word (bad count).
 *   k_new [B, max_new, dk]  v_new [B, max_new, dv]  kidx_new [B, max_new, dI]  n_new [B]
 *   k_main [B, N, dk]  v_main [B, N, dv]  k_idx [B, N, dI]  kb [B, ceil(N / block), dI] or NULL
 *   n_valid [B] (read and updated)
 * The caches, kb and n_valid are updated in place; ws holds only the error word. */
int csa2_kv_append(const csa2_shape* shape, int32_t max_new, const int32_t* n_new, const void* k_new,
                   const void* v_new, const void* kidx_new, void* k_main, void* v_main, void* k_idx, void* kb,
                   int32_t* n_valid, int32_t round_to_int, void* ws, size_t ws_bytes, csa2_stream_t stream);

/* One layer's part of csa2_swa_append. */
typedef struct {
  const void* k_tok;   /* [B, dk] the layer's key of the new token */
  const void* v_tok;   /* [B, dv] the layer's value of the new token */
  void* k_swa;         /* [B, W, dk] the layer's SWA ring (updated in place) */
  void* v_swa;         /* [B, W, dv] */
} csa2_swa_slot;

/* Decode-step cache maintenance, SWA windows (architecture page, bullet
 * "Sparse attention": every query also attends its last W tokens
 * uncompressed; mode table: every layer has its own SWA KV).
 * The layers of a group keep their windows as rings that share one head and
 * one fill count per query: for every layer l and query b, row swa_head[b] of
 * layers[l].k_swa[b] / v_swa[b] takes layers[l].k_tok[b] / v_tok[b]; then
 * swa_head[b] advances by one modulo W and n_swa[b] grows by one up to W.
 * Attention uses rows 0..n_swa[b]-1 as a set, so a ring needs no reordering.
 * A swa_head or n_swa outside 0..W-1 / 0..W is clamped and recorded in the
 * device error word (bad count).  1 <= n_layers <= 64; shape.swa >= 1.
 *   swa_head [B], n_swa [B] (read and updated) */
int csa2_swa_append(const csa2_shape* shape, const csa2_swa_slot* layers, int32_t n_layers, int32_t* swa_head,
                    int32_t* n_swa, void* ws, size_t ws_bytes, csa2_stream_t stream);

/* Hierarchical first stage: score every valid block summary key with the
 * indexer formula and keep the top min(P, NB_b) blocks, NB_b = ceil(n_valid[b] / block),
 * under (block score descending, block id ascending).
 *   q_idx [B, HI, dI]   w [B, HI]   kb [B, ceil(N / block), dI]   n_valid [B]
 *   pool_out   [B, P]  (output) pooled block ids in ascending order, padded with -1
 *   n_pool_out [B]     (output) min(P, NB_b) */
int csa2_index_blocks(const csa2_shape* shape, const void* q_idx, const float* w, const void* kb,
                      const int32_t* n_valid, int32_t* pool_out, int32_t* n_pool_out, void* ws,
                      size_t ws_bytes, csa2_stream_t stream);

/* Token-level indexer scores.
 * Flat (pool == NULL): scores_out[b, j] = s(k_idx[b, j]) for j < n_valid[b];
 *   cand_out (nullable) receives j; n_cand_out (nullable) receives n_valid[b].
 *   scores_out / cand_out have row stride N.
 * Pooled (pool != NULL, from csa2_index_blocks): the candidates are the
 *   entries of the pooled blocks in pool order (ascending entry id);
 *   position p*block + t holds entry pool[b, p]*block + t, its score, or
 *   cand -1 / score -inf when that entry is >= n_valid[b].
 *   scores_out / cand_out have row stride P*block; n_cand_out[b] = n_pool[b]*block.
 *   cand_out and n_cand_out are required. */
int csa2_index_tokens(const csa2_shape* shape, const void* q_idx, const float* w, const void* k_idx,
                      const int32_t* n_valid, const int32_t* pool, const int32_t* n_pool,
                      float* scores_out, int32_t* cand_out, int32_t* n_cand_out, void* ws,
                      size_t ws_bytes, csa2_stream_t stream);

/* Token scoring and exact Top-k in one call: the candidates of
 * csa2_index_tokens (flat when pool == NULL, else the pooled blocks' entries)
 * are scored and the top k (1 <= k <= shape.topk) selected under (score
 * descending, entry index ascending), as csa2_index_tokens followed by
 * csa2_topk would -- bullet "Sparse attention" (Top-512) and bullet
 * "Hierarchical indexer" (at most 16,384 pooled candidates).  On the fast
 * path (bf16, 8 x 64 indexer, blocks of 8) one thread-block cluster per query
 * scores its candidates and selects in shared memory without writing scores
 * to HBM.
 *   q_idx [B, HI, dI]  w [B, HI]  k_idx [B, N, dI]  n_valid [B]
 *   pool [B, P], n_pool [B] (from csa2_index_blocks) or NULL
 *   idx_out [B, k] (output) selected entry ids ascending, padded with -1
 *   n_out   [B]    (output, nullable) number selected */
int csa2_index_topk(const csa2_shape* shape, const void* q_idx, const float* w, const void* k_idx,
                    const int32_t* n_valid, const int32_t* pool, const int32_t* n_pool, int32_t k,
                    int32_t* idx_out, int32_t* n_out, void* ws, size_t ws_bytes, csa2_stream_t stream);

/* Exact Top-k of each row: scores [B, ld] (row stride ld), optional candidate
 * ids cand [B, ld] (NULL: the id is the position; ids < 0 are skipped; ids
 * must ascend with position), n_cand [B] positions to consider (NULL: ld).
 * Order: score descending, id ascending; -0 equals +0 and NaN ranks as -inf.
 *   idx_out   [B, k] (output) selected ids in ascending order, padded with -1
 *   score_out [B, k] (output, nullable) their scores (-inf for padding)
 * 1 <= k <= 16384, ld <= 2^28. */
int csa2_topk(const csa2_shape* shape, const float* scores, int32_t ld, const int32_t* cand,
              const int32_t* n_cand, int32_t k, int32_t* idx_out, float* score_out, void* ws,
              size_t ws_bytes, csa2_stream_t stream);

/* Sparse attention of one decode query per sequence (all H heads share one
 * KV head): one softmax over the main-KV rows idx[b, :] (entries < 0 are
 * skipped) and the SWA rows 0..n_swa[b]-1.
 *   q [B, H, dk]  k_main [B, N, dk]  v_main [B, N, dv]  idx [B, K]
 *   k_swa [B, W, dk]  v_swa [B, W, dv]  n_swa [B] (0..W)
 *   out [B, H, dv] (output)  lse [B, H] (output, nullable; -inf and out = 0
 *   when a query attends no row at all). */
int csa2_sparse_attn(const csa2_shape* shape, const void* q, const void* k_main, const void* v_main,
                     const int32_t* idx, const void* k_swa, const void* v_swa, const int32_t* n_swa,
                     float* out, float* lse, void* ws, size_t ws_bytes, csa2_stream_t stream);

/* A whole layer group over one shared main KV and indexer-key cache (the
 * group's Full layer's): layers run in order; Full and Reindex compute fresh
 * indices (flat, or hierarchical when layer.hier), Reuse attends with the
 * latest indices; every layer attends with its own q and SWA KV; an SWA
 * layer attends its SWA rows only.
 * Rules: a Reuse layer needs an earlier Full or Reindex layer in the group;
 * hier needs kb (from csa2_block_keys) and pool_blocks > 0.
 *   k_main [B, N, dk]  v_main [B, N, dv]  k_idx [B, N, dI]
 *   kb [B, ceil(N / block), dI] (nullable when no layer is hierarchical)
 *   n_valid [B] (0..N)  n_swa [B] (0..W) */
int csa2_layer_group(const csa2_shape* shape, const csa2_layer* layers, int32_t n_layers,
                     const void* k_main, const void* v_main, const void* k_idx, const void* kb,
                     const int32_t* n_valid, const int32_t* n_swa, void* ws, size_t ws_bytes,
                     csa2_stream_t stream);

/* csa2_layer_group for callers that cannot allocate device memory -- the
 * paper has no counterpart; this is a convenience of this library.  Some
 * callers have no way to provide a workspace: a plugin inside a host framework
 * that owns all device memory and exposes no allocator, or a latency-critical
 * decode loop that must not call cudaMalloc (it can synchronise the device).
 * This entry point takes the same arguments as csa2_layer_group minus the
 * workspace, and runs the same layer group on a 32 MiB scratch array that the
 * library holds in device memory (a file-scope __device__ array: every GPU
 * that loads the library keeps it until the process exits; it starts zeroed).
 *   - Shapes whose csa2_workspace_bytes exceeds 32 MiB return
 *     CSA2_ERR_WORKSPACE and enqueue nothing.
 *   - The first call made while a device is current looks up the array's
 *     device address (once per device, safe against host threads making
 *     their first calls at the same time); make that first call before any
 *     stream capture.
 *   - Every call shares the one array: calls that may overlap on the GPU (on
 *     different streams, or from different host threads without ordering)
 *     race on it and must be serialised by the caller.
 *   - No memory is allocated or freed.  Device-side range problems are
 *     skipped by the kernels as in csa2_layer_group and recorded in the
 *     array's header; read them with csa2_read_static_device_error.
 *   - kb can be prepared without a workspace too: csa2_block_keys and
 *     csa2_kv_append accept ws = NULL, ws_bytes = 0. */
int csa2_layer_group_static(const csa2_shape* shape, const csa2_layer* layers, int32_t n_layers,
                            const void* k_main, const void* v_main, const void* k_idx, const void* kb,
                            const int32_t* n_valid, const int32_t* n_swa, csa2_stream_t stream);

/* csa2_read_device_error for the static scratch array of the current device
 * (the error word of csa2_layer_group_static and of cache-maintenance calls
 * made with ws = NULL): synchronises `stream`, returns and clears the word.
 * The paper has no counterpart. */
int csa2_read_static_device_error(csa2_stream_t stream, int32_t* detail);

/* ---------------------------------------------------------------- context parallelism
 * One long sequence per query split over G ranks by block-aligned entry
 * ranges: rank g holds entries [e0_g, e0_g + n_loc_g) of every sequence.  The
 * pages describe no multi-GPU scheme; the split keeps the method's results
 * because its selection order (score descending, id ascending) is a strict
 * total order -- the Top-k of a union is the Top-k of the union of the parts'
 * Top-k lists -- and softmax partials over disjoint key sets combine exactly by
 * their log-sum-exp.  It serves contexts beyond one GPU, which the
 * architecture page's bullet "Hierarchical indexer" (at most 16,384
 * candidates whatever the context length) makes cheap to select over.  The
 * ranks exchange (score, id) lists and (out, lse) partials with their own
 * collectives; these calls are the per-rank steps around the exchanges. */

/* Keep the ids of each row that fall in [lo, hi), in their order, add delta,
 * and write them compacted to out[b, 0 .. n) with -1 after (n_out[b] = n).
 * Used both ways: a rank's local ids to global (lo = 0, hi = n_loc,
 * delta = e0) and a global list to a rank's local ids (lo = e0,
 * hi = e0 + n_loc, delta = -e0).  ids < 0 are dropped.  When a row keeps more
 * than ld_out ids the rest are dropped and the device error word records a
 * bad count.
 *   ids [batch, ld]   out [batch, ld_out]   n_out [batch] (nullable)
 *   ws: only its 256-byte header (error word) is used. */
int csa2_shard_slice(const int32_t* ids, int32_t batch, int32_t ld, int32_t lo, int32_t hi, int32_t delta,
                     int32_t* out, int32_t ld_out, int32_t* n_out, void* ws, size_t ws_bytes, csa2_stream_t stream);

/* A rank's valid entries (div = 1) or valid blocks (div = block) per query:
 * out[b] = ceil(clamp(n_valid[b] - e0, 0, n_loc) / div).
 *   n_valid [batch] (global counts)   out [batch] */
int csa2_shard_counts(const int32_t* n_valid, int32_t batch, int32_t e0, int32_t n_loc, int32_t div, int32_t* out,
                      csa2_stream_t stream);

/* The G parts' (id, score) lists of every row side by side, in part order:
 * ids_out[b, g*k + p] = ids[g, b, p] and likewise for the scores (nullable),
 * turning the [parts, batch, k] result of an all-gather into the [batch,
 * parts*k] candidate rows of csa2_topk. */
int csa2_concat_parts(int32_t parts, int32_t batch, int32_t k, const int32_t* ids, const float* scores,
                      int32_t* ids_out, float* scores_out, csa2_stream_t stream);

/* Combine the softmax attention of `parts` disjoint key sets, in part order:
 * with M = max_g lse_g and w_g = exp(lse_g - M),
 *   out = sum_g w_g out_g / sum_g w_g,   lse = M + log(sum_g w_g);
 * parts with lse = -inf (no key) contribute nothing; all -inf gives out = 0
 * and lse = -inf.  Rows are (query, head) pairs.
 *   out_parts [parts, rows, v_dim]  lse_parts [parts, rows] (natural log)
 *   out [rows, v_dim]  lse [rows] (nullable) */
int csa2_merge_attn(int32_t parts, int32_t rows, int32_t v_dim, const float* out_parts, const float* lse_parts,
                    float* out, float* lse, csa2_stream_t stream);

/* Static description of a status code. */
const char* csa2_status_str(int status);

/* Synchronise `stream`, read and clear the sticky device error word of `ws`.
 * Returns CSA2_OK, CSA2_ERR_DEVICE_CHECK or CSA2_ERR_TIMEOUT (a bounded wait
 * gave up); *detail (nullable) receives the error bits (bit 0 bad index,
 * bit 1 bad count, bit 2 timeout, bit 3 bad pooled block) in its low byte. */
int csa2_read_device_error(void* ws, csa2_stream_t stream, int32_t* detail);

/* 1 when the fast (tensor-core) kernels serve this shape, 0 when the generic
 * kernels do (host only; for diagnostics and tests). */
int csa2_fast_path(const csa2_shape* shape, int32_t* indexer_fast, int32_t* attention_fast);

/* Number of kernel launches this library has enqueued since it was loaded
 * (all threads and devices; launches recorded into a CUDA graph count once,
 * at capture).  For diagnostics and launch accounting. */
unsigned long long csa2_launch_count(void);

/* Test hook of the device-side failure detection (diagnostics; the paper has
 * no counterpart).  Runs the fused flat scoring + Top-k of csa2_index_topk
 * (pool == NULL; fast path only, else CSA2_ERR_UNSUPPORTED) with the copy of
 * every CTA's first key tile left out, so that the tile's stage barrier can
 * never complete, and with every bounded wait limited to wait_limit_ns
 * (1,000 .. 100,000,000) instead of 2 s.  The waits give up, the kernel
 * records CSA2_ERR_TIMEOUT (bit 2) in the workspace's error word, the CTAs
 * that gave up offer no candidate, and the kernel returns: no copy is in
 * flight when a wait gives up and every write stays inside idx_out [B, k].
 * csa2_read_device_error then returns CSA2_ERR_TIMEOUT, and the stream and
 * context stay usable. */
int csa2_debug_wait_timeout(const csa2_shape* shape, const void* q_idx, const float* w, const void* k_idx,
                            const int32_t* n_valid, int32_t k, int32_t* idx_out, uint32_t wait_limit_ns,
                            void* ws, size_t ws_bytes, csa2_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CSA2_H_ */

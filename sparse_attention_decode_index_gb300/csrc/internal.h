// Internal interface between the C-ABI host code (api.cu) and the kernel
// translation units.  Not installed; not part of the public ABI.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace csa2 {

// Bits of the sticky device error word (word 0 of the workspace header).
constexpr int kErrBadIndex = 1;   // a main-KV index outside [0, n_entries)
constexpr int kErrBadCount = 2;   // n_valid / n_swa / n_pool / n_cand outside its range
constexpr int kErrTimeout = 4;    // a bounded wait on an mbarrier gave up
constexpr int kErrBadPool = 8;    // a pooled block id outside [0, ceil(n_valid / block))

// Indexer scoring: s = sum_h w_h * ReLU(q_h . k) over a flat row range or the
// entries of pooled blocks.
struct IndexerArgs {
  const void* keys;          // [B / seq_div, rows_per_seq, dim] (indexer keys or block keys)
  long long rows_per_seq;    // row capacity per sequence
  int seq_div;               // queries per key sequence: query b reads sequence b / seq_div
  const void* q_idx;         // [B, heads, dim]
  const float* w;            // [B, heads]
  const int* n_valid;        // [B] valid compressed entries per query
  int valid_cap;             // capacity n_valid is checked against
  int div;                   // flat: valid rows = ceil(n_valid / div) (1 or block)
  const int* pool;           // pooled: [B, pool_cap] ascending block ids
  const int* n_pool;         // pooled: [B]
  int pool_cap;              // pooled: row stride of `pool`
  int block;                 // entries per block
  float* scores;             // [B, ld]
  int* cand;                 // [B, ld] candidate entry ids (nullable when flat)
  int* n_cand;               // [B] candidate positions written (nullable)
  long long ld;              // row stride of scores / cand
  int per_cta;               // flat: rows per CTA; pooled: pool positions per CTA
  int relu;
  int heads, dim, dtype;     // generic kernel only
  int* err;                  // device error word (nullable)
};

struct TopkArgs {
  const float* scores;       // row r = b * rows_per_b ... ; element (r, pos)
  long long ld_in;           // row stride of scores / cand
  const int* cand;           // nullable: id = position; entries < 0 are skipped
  const int* n_cand;         // [B] positions to consider (nullable -> n_fixed)
  int n_fixed;
  int n_cap;                 // n_cand is clamped to this
  int chunk;                 // positions per CTA (grid.x = chunks)
  int k;
  int* idx_out;              // [B, chunks, k]
  float* score_out;          // [B, chunks, k] (nullable)
  int* n_out;                // [B] number selected (nullable; single-chunk launches only)
  int* err;
};

struct AttnArgs {
  const void* q;             // [B, H, dk]
  const void* k_main;        // [B / seq_div, N, dk]
  const void* v_main;        // [B / seq_div, N, dv]
  int seq_div;               // queries per KV sequence: query b reads sequence b / seq_div
  const int* idx;            // [B, topk]
  const void* k_swa;         // [B, W, dk]
  const void* v_swa;         // [B, W, dv]
  const int* n_swa;          // [B]
  float* out;                // [B, H, dv]
  float* lse;                // [B, H] (nullable)
  int n_entries, topk, swa;
  int heads, k_dim, v_dim, dtype;
  float scale;               // softmax scale (natural-log domain)
  int* err;
  int release_at_end;        // fast path: let the next launch place its CTAs only at this one's end
};

// Fused scoring + cluster Top-k (fused.cu): one cluster per query scores its
// candidates and writes the selected ids (ascending, -1 padded).
struct SelectArgs {
  const void* keys;          // [B / seq_div, rows_per_seq, 64] bf16 (indexer keys or block keys)
  long long rows_per_seq;
  int seq_div;               // queries per key sequence: query b reads sequence b / seq_div
  const void* q_idx;         // [B, 8, 64] bf16
  const float* w;            // [B, 8]
  int relu;
  const int* n_valid;        // [B]
  int valid_cap;
  int div;                   // flat: candidates = ceil(n_valid / div)
  const int* pool;           // pooled: [B, pool_cap] ascending block ids
  const int* n_pool;         // pooled: [B]
  int pool_cap;
  int rows_per_cta;          // set by the launcher: rows (flat) / pool positions (pooled) per CTA
  int k;                     // how many to select
  int* out;                  // [B, ld_out] selected ids
  long long ld_out;
  int* n_out;                // [B] number selected (nullable)
  int* err;
  // Test hooks of the bounded waits (0 in every production launch): a limit
  // for every mbarrier wait instead of the default 2 s, and a flag that
  // leaves out the copy of each CTA's first tile, so that the tile's stage
  // barrier cannot complete and the waits run out (no copy is in flight
  // when they give up).
  unsigned long long wait_ns;
  int skip_first_copy;
};

bool index_select_supported(bool pooled, int max_units);
cudaError_t launch_index_select(const SelectArgs& a, bool pooled, int batch, int max_units, cudaStream_t st);

struct BlockKeyArgs {
  const void* k_idx;         // [B / seq_div, N, dim]
  const int* n_valid;        // [B] (per query)
  void* kb;                  // [B, NB, dim] (per query)
  int seq_div;               // queries per key sequence
  int n_entries, nb_cap, dim, block, round_to_int, dtype;
  int* err;
};

// Decode-step cache maintenance (append.cu).
struct KvAppendArgs {
  const int* n_new;          // [B]
  int max_new;
  const void* k_new;         // [B, max_new, k_dim]
  const void* v_new;         // [B, max_new, v_dim]
  const void* kidx_new;      // [B, max_new, idx_dim]
  void* k_main;              // [B, N, k_dim]
  void* v_main;              // [B, N, v_dim]
  void* k_idx;               // [B, N, idx_dim]
  void* kb;                  // [B, nb_cap, idx_dim] or null
  int* n_valid;              // [B] (read and updated)
  int n_entries, nb_cap, k_dim, v_dim, idx_dim, block, round_to_int, dtype;
  int* err;
};

constexpr int kMaxSwaLayers = 64;

struct SwaAppendArgs {
  struct Slot {
    const void* k_tok;       // [B, k_dim]
    const void* v_tok;       // [B, v_dim]
    void* k_swa;             // [B, W, k_dim]
    void* v_swa;             // [B, W, v_dim]
  } slot[kMaxSwaLayers];
  int n_layers;
  int* head;                 // [B] (read and updated)
  int* n_swa;                // [B] (read and updated)
  int swa, k_dim, v_dim, dtype;
  int* err;
};

// Context-parallel helpers (shard.cu).
struct ShardSliceArgs {
  const int* ids;            // [B, ld] ids (ascending in the uses here; -1 and ids outside [lo, hi) are dropped)
  long long ld;
  int lo, hi, delta;
  int* out;                  // [B, ld_out] kept ids + delta in input order, -1 padded
  long long ld_out;
  int* n_out;                // [B] kept count (nullable)
  int* err;
};

struct MergeAttnArgs {
  const float* out_parts;    // [parts, rows, v_dim]
  const float* lse_parts;    // [parts, rows]
  float* out;                // [rows, v_dim]
  float* lse;                // [rows] (nullable)
  int parts, rows, v_dim;
};

cudaError_t launch_shard_slice(const ShardSliceArgs& a, int batch, cudaStream_t st);
struct ConcatArgs {
  const int* ids;            // [parts, batch, k]
  const float* scores;       // [parts, batch, k] (nullable)
  int* ids_out;              // [batch, parts * k]
  float* scores_out;         // [batch, parts * k] (written when scores is not null)
  int parts, batch, k;
};

cudaError_t launch_shard_counts(const int* n_valid, int batch, int e0, int n_loc, int div, int* out,
                                cudaStream_t st);
cudaError_t launch_concat_parts(const ConcatArgs& a, cudaStream_t st);
cudaError_t launch_merge_attn(const MergeAttnArgs& a, cudaStream_t st);

cudaError_t launch_kv_append(const KvAppendArgs& a, int batch, cudaStream_t st);
cudaError_t launch_swa_append(const SwaAppendArgs& a, int batch, cudaStream_t st);

int device_sm_count();

// Device address of the library's static scratch array (static_ws.cu) on the
// current device, looked up once per device; CSA2_OK or CSA2_ERR_CUDA.
int static_scratch(void** out);

// Launch `kernel` with programmatic stream serialization (PDL) and an optional
// cluster shape; every kernel of the library calls pdl_wait() before touching
// data of earlier launches.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       unsigned cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}
// Counts kernel launches enqueued by the library (diagnostics: csa2_launch_count).
void note_launch();

// Per-device one-time set-up (a kernel's shared-memory opt-in is a per-device
// attribute): runs `set` with the current device current the first time `key`
// (0..63) is seen on that device, and again until it succeeds.  Thread-safe.
enum SetupKey { kSetupAttn = 0, kSetupIndexerFlat = 1, kSetupIndexerPooled = 2, kSetupSelectFlat = 3,
                kSetupSelectPooled = 4 };
cudaError_t once_per_device(int key, cudaError_t (*set)());

cudaError_t launch_block_keys(const BlockKeyArgs& a, int batch, cudaStream_t st);
// fast: bf16, 8 heads x 64 dims, block 8 (pooled)
cudaError_t launch_indexer(const IndexerArgs& a, bool pooled, bool fast, int batch, int max_rows,
                           cudaStream_t st);
cudaError_t launch_topk(const TopkArgs& a, int chunks, int batch, cudaStream_t st);
int topk_max_chunk();
// Cluster Top-k over one row of up to topk_cluster_max() positions (one launch).
cudaError_t launch_topk_cluster(const TopkArgs& a, int batch, cudaStream_t st);
int topk_cluster_max();
// Cluster size of the fast attention kernel for these slot counts (0: unsupported).
int attn_cluster(int topk, int swa);
// fast: bf16, 64 heads, dk 192, dv 128
cudaError_t launch_attn(const AttnArgs& a, bool fast, int batch, cudaStream_t st);

}  // namespace csa2

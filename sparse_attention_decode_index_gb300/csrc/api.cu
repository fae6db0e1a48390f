// Host side of the C ABI declared in include/csa2.h: argument validation,
// workspace carving, kernel selection and the layer-group sequencing.
//
// Layer-group sequencing follows the mode table of the DeepSeek V4.1 Flash
// architecture page ("CSA2 with cross-layer reuse"): Full and Reindex layers
// compute fresh Top-K indices over the group's shared indexer keys (Reindex
// with its own indexer query), Reuse layers attend with the latest indices,
// and every layer attends with its own query and SWA KV.
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/csa2.h"
#include "internal.h"

using namespace csa2;

namespace csa2 {
static std::atomic<unsigned long long> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

constexpr int kMaxSetupDevices = 64;
static std::atomic<uint64_t> g_setup_done[kMaxSetupDevices];
static std::mutex g_setup_mu;

cudaError_t once_per_device(int key, cudaError_t (*set)()) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxSetupDevices || key < 0 || key >= 64) return set();
  const uint64_t bit = uint64_t(1) << key;
  if (g_setup_done[dev].load(std::memory_order_acquire) & bit) return cudaSuccess;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_setup_done[dev].load(std::memory_order_relaxed) & bit) return cudaSuccess;
  e = set();
  if (e == cudaSuccess) g_setup_done[dev].fetch_or(bit, std::memory_order_release);
  return e;
}
}  // namespace csa2

namespace {

constexpr size_t kAlign = 256;
constexpr size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct WsLayout {
  size_t hdr, pool, n_pool, n_blk, blk_scores, tok_scores, tok_cand, n_cand, tk_ids_a, tk_sc_a, tk_ids_b,
      tk_sc_b, idx, total;
  int64_t nb_cap, tok_ld, tk_chunks, tk_kmax;
};

bool hier_possible(const csa2_shape& s) { return s.pool_blocks > 0; }
bool attn_fast(const csa2_shape& s);

WsLayout layout(const csa2_shape& s) {
  WsLayout L{};
  const int64_t B = s.batch;
  L.nb_cap = ceil_div(s.n_entries, s.block);
  const int64_t P = hier_possible(s) ? s.pool_blocks : 0;
  L.tok_ld = s.n_entries > P * s.block ? s.n_entries : P * s.block;
  const int64_t longest = L.tok_ld > L.nb_cap ? L.tok_ld : L.nb_cap;
  const int64_t maxc = topk_max_chunk();
  L.tk_kmax = s.topk > P ? s.topk : P;
  L.tk_chunks = longest > maxc ? ceil_div(longest, maxc) : 0;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes);
    return at;
  };
  L.hdr = take(256);
  L.pool = take(size_t(B * P) * 4);
  L.n_pool = take(size_t(B) * 4);
  L.n_blk = take(size_t(B) * 4);
  L.blk_scores = take(size_t(B * L.nb_cap) * 4);
  L.tok_scores = take(size_t(B * L.tok_ld) * 4);
  L.tok_cand = take(size_t(B * L.tok_ld) * 4);
  L.n_cand = take(size_t(B) * 4);
  const size_t tk = size_t(B * L.tk_chunks * L.tk_kmax) * 4;
  L.tk_ids_a = take(tk);
  L.tk_sc_a = take(tk);
  L.tk_ids_b = take(tk);
  L.tk_sc_b = take(tk);
  L.idx = take(size_t(B) * s.topk * 4);
  L.total = off;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

#define CSA2_TRY(x)                   \
  do {                                \
    const int _st = (x);              \
    if (_st != CSA2_OK) return _st;   \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(const csa2_shape* s) {
  if (s == nullptr) return CSA2_ERR_INVALID_ARG;
  if (s->batch < 1 || s->n_entries < 1 || s->idx_heads < 1 || s->idx_dim < 1 || s->block < 1 ||
      s->pool_blocks < 0 || s->topk < 1 || s->q_heads < 1 || s->k_dim < 1 || s->v_dim < 1 || s->swa < 0)
    return CSA2_ERR_INVALID_ARG;
  if (s->dtype != CSA2_BF16 && s->dtype != CSA2_F32) return CSA2_ERR_INVALID_ARG;
  if (s->relu != 0 && s->relu != 1) return CSA2_ERR_INVALID_ARG;
  if (s->tokens < 0 || (s->tokens > 1 && s->batch % s->tokens != 0)) return CSA2_ERR_INVALID_ARG;
  if (s->n_entries > (1 << 28) || s->batch > (1 << 20)) return CSA2_ERR_UNSUPPORTED;
  if (s->idx_heads > 64 || s->idx_dim > 1024 || s->idx_heads * s->idx_dim > 8192) return CSA2_ERR_UNSUPPORTED;
  if (s->topk > 1024 || s->swa > 1024 || s->topk + s->swa > 1024) return CSA2_ERR_UNSUPPORTED;
  if (s->q_heads > 1024 || s->k_dim > 1024 || s->v_dim > 1024) return CSA2_ERR_UNSUPPORTED;
  if (int64_t(s->pool_blocks) * s->block > (1 << 24)) return CSA2_ERR_UNSUPPORTED;
  if (s->pool_blocks > topk_max_chunk() / 2) return CSA2_ERR_UNSUPPORTED;
  return CSA2_OK;
}

// Queries per cache sequence (csa2_shape.tokens; 0 means 1).
int seqdiv(const csa2_shape& s) { return s.tokens > 1 ? s.tokens : 1; }

bool indexer_fast(const csa2_shape& s) { return s.dtype == CSA2_BF16 && s.idx_heads == 8 && s.idx_dim == 64; }
bool pooled_fast(const csa2_shape& s) { return indexer_fast(s) && s.block == 8; }
bool attn_fast(const csa2_shape& s) {
  return s.dtype == CSA2_BF16 && s.q_heads == 64 && s.k_dim == 192 && s.v_dim == 128 &&
         attn_cluster(s.topk, s.swa) > 0;
}

int check_ws(const csa2_shape& s, void* ws, size_t bytes) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return CSA2_ERR_WORKSPACE;
  if (bytes < layout(s).total) return CSA2_ERR_WORKSPACE;
  return CSA2_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA; }

// Device error word of a cache-maintenance call: the header of the caller's
// workspace, or, when the caller passes no workspace (ws NULL, ws_bytes 0),
// the header of the library's static scratch array on the current device.
int error_word(const csa2_shape& s, void* ws, size_t ws_bytes, int** err) {
  if (ws == nullptr && ws_bytes == 0) {
    void* p = nullptr;
    CSA2_TRY(static_scratch(&p));
    *err = static_cast<int*>(p);
    return CSA2_OK;
  }
  CSA2_TRY(check_ws(s, ws, ws_bytes));
  *err = static_cast<int*>(ws);
  return CSA2_OK;
}

float softmax_scale(const csa2_shape& s) { return s.scale > 0.f ? s.scale : 1.0f / sqrtf(float(s.k_dim)); }

// ---------------------------------------------------------------- internal ops (no validation)

int do_index_flat(const csa2_shape& s, const void* q_idx, const float* w, const void* keys, int64_t rows_per_seq, int seq_div,
                  const int32_t* n_valid, int div, float* scores, int32_t* cand, int32_t* n_cand, int64_t ld,
                  int* err, cudaStream_t st) {
  IndexerArgs a{};
  a.keys = keys;
  a.rows_per_seq = rows_per_seq;
  a.seq_div = seq_div;
  a.q_idx = q_idx;
  a.w = w;
  a.n_valid = n_valid;
  a.valid_cap = s.n_entries;
  a.div = div;
  a.block = s.block;
  a.scores = scores;
  a.cand = cand;
  a.n_cand = n_cand;
  a.ld = ld;
  a.relu = s.relu;
  a.heads = s.idx_heads;
  a.dim = s.idx_dim;
  a.dtype = s.dtype;
  a.err = err;
  const int max_rows = int(ceil_div(s.n_entries, div));
  return cuda_status(launch_indexer(a, false, indexer_fast(s), s.batch, max_rows, st));
}

int do_index_pooled(const csa2_shape& s, const void* q_idx, const float* w, const void* k_idx,
                    const int32_t* n_valid, const int32_t* pool, const int32_t* n_pool, float* scores,
                    int32_t* cand, int32_t* n_cand, int* err, cudaStream_t st) {
  IndexerArgs a{};
  a.keys = k_idx;
  a.rows_per_seq = s.n_entries;
  a.seq_div = seqdiv(s);
  a.q_idx = q_idx;
  a.w = w;
  a.n_valid = n_valid;
  a.valid_cap = s.n_entries;
  a.div = 1;
  a.pool = pool;
  a.n_pool = n_pool;
  a.pool_cap = s.pool_blocks;
  a.block = s.block;
  a.scores = scores;
  a.cand = cand;
  a.n_cand = n_cand;
  a.ld = int64_t(s.pool_blocks) * s.block;
  a.relu = s.relu;
  a.heads = s.idx_heads;
  a.dim = s.idx_dim;
  a.dtype = s.dtype;
  a.err = err;
  return cuda_status(launch_indexer(a, true, pooled_fast(s), s.batch, s.pool_blocks, st));
}

// Exact Top-k: rows longer than one cluster can hold are first cut into chunks
// of <= topk_max_chunk() positions whose Top-k lists are merged, then one
// cluster launch selects the final Top-k.
int do_topk(const csa2_shape& s, const WsLayout& L, void* ws, const float* scores, int64_t ld,
            const int32_t* cand, const int32_t* n_cand, int64_t n_cap, int k, int32_t* idx_out,
            float* score_out, int32_t* n_out, cudaStream_t st) {
  int* err = at<int>(ws, L.hdr);
  const int64_t maxc = topk_max_chunk();
  const int64_t maxcl = topk_cluster_max();
  TopkArgs a{};
  a.scores = scores;
  a.ld_in = ld;
  a.cand = cand;
  a.n_cand = n_cand;
  a.n_fixed = int(n_cap);
  a.n_cap = int(n_cap);
  a.k = k;
  a.err = err;
  int64_t n = n_cap;
  bool use_a = true;
  while (n > maxcl) {
    const int64_t chunks = ceil_div(n, maxc);
    a.chunk = int(ceil_div(n, chunks));
    a.idx_out = at<int32_t>(ws, use_a ? L.tk_ids_a : L.tk_ids_b);
    a.score_out = at<float>(ws, use_a ? L.tk_sc_a : L.tk_sc_b);
    a.n_out = nullptr;
    CSA2_TRY(cuda_status(launch_topk(a, int(chunks), s.batch, st)));
    // next level reads the concatenated chunk lists
    n = chunks * k;
    a.scores = a.score_out;
    a.cand = a.idx_out;
    a.ld_in = n;
    a.n_cand = nullptr;
    a.n_fixed = int(n);
    a.n_cap = int(n);
    use_a = !use_a;
  }
  a.n_cap = int(n > 0 ? n : 1);
  if (a.n_cand == nullptr) a.n_fixed = int(n);
  a.idx_out = idx_out;
  a.score_out = score_out;
  a.n_out = n_out;
  return cuda_status(launch_topk_cluster(a, s.batch, st));
}

int do_attn(const csa2_shape& s, const void* q, const void* k_main, const void* v_main, const int32_t* idx,
            const void* k_swa, const void* v_swa, const int32_t* n_swa, float* out, float* lse, int* err,
            cudaStream_t st, bool swa_only = false, bool release_at_end = false) {
  AttnArgs a{};
  a.release_at_end = release_at_end ? 1 : 0;
  a.q = q;
  a.k_main = k_main;
  a.v_main = v_main;
  a.seq_div = seqdiv(s);
  a.idx = idx;
  a.k_swa = k_swa;
  a.v_swa = v_swa;
  a.n_swa = n_swa;
  a.out = out;
  a.lse = lse;
  a.n_entries = s.n_entries;
  a.topk = swa_only ? 0 : s.topk;   // a pure SWA layer has no main-KV slots
  a.swa = s.swa;
  a.heads = s.q_heads;
  a.k_dim = s.k_dim;
  a.v_dim = s.v_dim;
  a.dtype = s.dtype;
  a.scale = softmax_scale(s);
  a.err = err;
  return cuda_status(launch_attn(a, attn_fast(s), s.batch, st));
}

SelectArgs select_args(const csa2_shape& s, const void* keys, int64_t rows_per_seq, int seq_div, const void* q_idx,
                       const float* w, const int32_t* n_valid, int div, int k, int32_t* out, int64_t ld_out,
                       int32_t* n_out, int* err) {
  SelectArgs a{};
  a.keys = keys;
  a.rows_per_seq = rows_per_seq;
  a.seq_div = seq_div;
  a.q_idx = q_idx;
  a.w = w;
  a.relu = s.relu;
  a.n_valid = n_valid;
  a.valid_cap = s.n_entries;
  a.div = div;
  a.k = k;
  a.out = out;
  a.ld_out = ld_out;
  a.n_out = n_out;
  a.err = err;
  return a;
}

int do_index_blocks(const csa2_shape& s, const WsLayout& L, void* ws, const void* q_idx, const float* w,
                    const void* kb, const int32_t* n_valid, int32_t* pool_out, int32_t* n_pool_out,
                    cudaStream_t st) {
  int* err = at<int>(ws, L.hdr);
  if (indexer_fast(s) && index_select_supported(false, int(L.nb_cap))) {
    // fused: block scoring and pool selection in one cluster launch
    SelectArgs a = select_args(s, kb, L.nb_cap, 1, q_idx, w, n_valid, s.block, s.pool_blocks, pool_out,
                               s.pool_blocks, n_pool_out, err);
    return cuda_status(launch_index_select(a, false, s.batch, int(L.nb_cap), st));
  }
  float* bs = at<float>(ws, L.blk_scores);
  int32_t* nblk = at<int32_t>(ws, L.n_blk);
  CSA2_TRY(do_index_flat(s, q_idx, w, kb, L.nb_cap, 1, n_valid, s.block, bs, nullptr, nblk, L.nb_cap, err, st));
  return do_topk(s, L, ws, bs, L.nb_cap, nullptr, nblk, L.nb_cap, s.pool_blocks, pool_out, nullptr, n_pool_out,
                 st);
}

int check_sswa(const csa2_shape& s, const void* k_swa, const void* v_swa, const int32_t* n_swa) {
  if (n_swa == nullptr) return CSA2_ERR_INVALID_ARG;
  if (s.swa > 0 && (k_swa == nullptr || v_swa == nullptr)) return CSA2_ERR_INVALID_ARG;
  if (attn_fast(s) && s.swa > 0 && (!aligned16(k_swa) || !aligned16(v_swa))) return CSA2_ERR_INVALID_ARG;
  return CSA2_OK;
}

int check_attn_args(const csa2_shape& s, const void* q, const void* k_main, const void* v_main, float* out) {
  if (q == nullptr || k_main == nullptr || v_main == nullptr || out == nullptr) return CSA2_ERR_INVALID_ARG;
  if (attn_fast(s) && (!aligned16(q) || !aligned16(k_main) || !aligned16(v_main))) return CSA2_ERR_INVALID_ARG;
  return CSA2_OK;
}

}  // namespace

// ====================================================================== C ABI

extern "C" {

size_t csa2_workspace_bytes(const csa2_shape* shape) {
  if (check_shape(shape) != CSA2_OK) return 0;
  return layout(*shape).total;
}

int csa2_workspace_init(void* ws, size_t ws_bytes, csa2_stream_t stream) {
  if (ws == nullptr || ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0)
    return CSA2_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, 256, stream));
}

int csa2_block_keys(const csa2_shape* shape, const void* k_idx, const int32_t* n_valid, int32_t round_to_int,
                    void* kb, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  CSA2_TRY(check_shape(shape));
  const csa2_shape& s = *shape;
  if (k_idx == nullptr || n_valid == nullptr || kb == nullptr) return CSA2_ERR_INVALID_ARG;
  if (round_to_int != 0 && round_to_int != 1) return CSA2_ERR_INVALID_ARG;
  int* err = nullptr;
  CSA2_TRY(error_word(s, ws, ws_bytes, &err));
  const WsLayout L = layout(s);
  BlockKeyArgs a{};
  a.k_idx = k_idx;
  a.seq_div = seqdiv(s);
  a.n_valid = n_valid;
  a.kb = kb;
  a.n_entries = s.n_entries;
  a.nb_cap = int(L.nb_cap);
  a.dim = s.idx_dim;
  a.block = s.block;
  a.round_to_int = round_to_int;
  a.dtype = s.dtype;
  a.err = err;
  return cuda_status(launch_block_keys(a, s.batch, stream));
}

int csa2_kv_append(const csa2_shape* shape, int32_t max_new, const int32_t* n_new, const void* k_new,
                   const void* v_new, const void* kidx_new, void* k_main, void* v_main, void* k_idx, void* kb,
                   int32_t* n_valid, int32_t round_to_int, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  CSA2_TRY(check_shape(shape));
  const csa2_shape& s = *shape;
  if (seqdiv(s) != 1) return CSA2_ERR_UNSUPPORTED;   // appends are per sequence: pass a one-token shape
  if (max_new < 0 || max_new > s.n_entries) return CSA2_ERR_INVALID_ARG;
  if (n_new == nullptr || n_valid == nullptr || k_main == nullptr || v_main == nullptr || k_idx == nullptr)
    return CSA2_ERR_INVALID_ARG;
  if (max_new > 0 && (k_new == nullptr || v_new == nullptr || kidx_new == nullptr)) return CSA2_ERR_INVALID_ARG;
  if (round_to_int != 0 && round_to_int != 1) return CSA2_ERR_INVALID_ARG;
  int* err = nullptr;
  CSA2_TRY(error_word(s, ws, ws_bytes, &err));
  const WsLayout L = layout(s);
  KvAppendArgs a{};
  a.n_new = n_new;
  a.max_new = max_new;
  a.k_new = k_new;
  a.v_new = v_new;
  a.kidx_new = kidx_new;
  a.k_main = k_main;
  a.v_main = v_main;
  a.k_idx = k_idx;
  a.kb = kb;
  a.n_valid = n_valid;
  a.n_entries = s.n_entries;
  a.nb_cap = int(L.nb_cap);
  a.k_dim = s.k_dim;
  a.v_dim = s.v_dim;
  a.idx_dim = s.idx_dim;
  a.block = s.block;
  a.round_to_int = round_to_int;
  a.dtype = s.dtype;
  a.err = err;
  return cuda_status(launch_kv_append(a, s.batch, stream));
}

int csa2_swa_append(const csa2_shape* shape, const csa2_swa_slot* layers, int32_t n_layers, int32_t* swa_head,
                    int32_t* n_swa, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  CSA2_TRY(check_shape(shape));
  const csa2_shape& s = *shape;
  if (seqdiv(s) != 1) return CSA2_ERR_UNSUPPORTED;   // rings are per query: pass a one-token shape
  if (s.swa < 1 || layers == nullptr || n_layers < 1 || n_layers > kMaxSwaLayers) return CSA2_ERR_INVALID_ARG;
  if (swa_head == nullptr || n_swa == nullptr) return CSA2_ERR_INVALID_ARG;
  int* err = nullptr;
  CSA2_TRY(error_word(s, ws, ws_bytes, &err));
  SwaAppendArgs a{};
  for (int l = 0; l < n_layers; ++l) {
    const csa2_swa_slot& y = layers[l];
    if (y.k_tok == nullptr || y.v_tok == nullptr || y.k_swa == nullptr || y.v_swa == nullptr)
      return CSA2_ERR_INVALID_ARG;
    a.slot[l] = SwaAppendArgs::Slot{y.k_tok, y.v_tok, y.k_swa, y.v_swa};
  }
  a.n_layers = n_layers;
  a.head = swa_head;
  a.n_swa = n_swa;
  a.swa = s.swa;
  a.k_dim = s.k_dim;
  a.v_dim = s.v_dim;
  a.dtype = s.dtype;
  a.err = err;
  return cuda_status(launch_swa_append(a, s.batch, stream));
}

int csa2_index_blocks(const csa2_shape* shape, const void* q_idx, const float* w, const void* kb,
                      const int32_t* n_valid, int32_t* pool_out, int32_t* n_pool_out, void* ws, size_t ws_bytes,
                      csa2_stream_t stream) {
  CSA2_TRY(check_shape(shape));
  const csa2_shape& s = *shape;
  CSA2_TRY(check_ws(s, ws, ws_bytes));
  if (s.pool_blocks < 1) return CSA2_ERR_INVALID_ARG;
  if (q_idx == nullptr || w == nullptr || kb == nullptr || n_valid == nullptr || pool_out == nullptr ||
      n_pool_out == nullptr)
    return CSA2_ERR_INVALID_ARG;
  if (indexer_fast(s) && !aligned16(kb)) return CSA2_ERR_INVALID_ARG;
  const WsLayout L = layout(s);
  return do_index_blocks(s, L, ws, q_idx, w, kb, n_valid, pool_out, n_pool_out, stream);
}

int csa2_index_tokens(const csa2_shape* shape, const void* q_idx, const float* w, const void* k_idx,
                      const int32_t* n_valid, const int32_t* pool, const int32_t* n_pool, float* scores_out,
                      int32_t* cand_out, int32_t* n_cand_out, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  CSA2_TRY(check_shape(shape));
  const csa2_shape& s = *shape;
  CSA2_TRY(check_ws(s, ws, ws_bytes));
  if (q_idx == nullptr || w == nullptr || k_idx == nullptr || n_valid == nullptr || scores_out == nullptr)
    return CSA2_ERR_INVALID_ARG;
  if (indexer_fast(s) && !aligned16(k_idx)) return CSA2_ERR_INVALID_ARG;
  const WsLayout L = layout(s);
  int* err = at<int>(ws, L.hdr);
  if (pool == nullptr)
    return do_index_flat(s, q_idx, w, k_idx, s.n_entries, seqdiv(s), n_valid, 1, scores_out, cand_out, n_cand_out,
                         s.n_entries, err, stream);
  if (s.pool_blocks < 1 || n_pool == nullptr || cand_out == nullptr || n_cand_out == nullptr)
    return CSA2_ERR_INVALID_ARG;
  if (s.n_entries % s.block != 0) return CSA2_ERR_INVALID_ARG;
  return do_index_pooled(s, q_idx, w, k_idx, n_valid, pool, n_pool, scores_out, cand_out, n_cand_out, err,
                         stream);
}

int csa2_index_topk(const csa2_shape* shape, const void* q_idx, const float* w, const void* k_idx,
                    const int32_t* n_valid, const int32_t* pool, const int32_t* n_pool, int32_t k, int32_t* idx_out,
                    int32_t* n_out, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  CSA2_TRY(check_shape(shape));
  const csa2_shape& s = *shape;
  CSA2_TRY(check_ws(s, ws, ws_bytes));
  if (q_idx == nullptr || w == nullptr || k_idx == nullptr || n_valid == nullptr || idx_out == nullptr || k < 1)
    return CSA2_ERR_INVALID_ARG;
  if (k > s.topk) return CSA2_ERR_INVALID_ARG;      // the workspace is sized for shape.topk
  if (indexer_fast(s) && !aligned16(k_idx)) return CSA2_ERR_INVALID_ARG;
  const WsLayout L = layout(s);
  int* err = at<int>(ws, L.hdr);
  float* ts = at<float>(ws, L.tok_scores);
  int32_t* tc = at<int32_t>(ws, L.tok_cand);
  int32_t* nc = at<int32_t>(ws, L.n_cand);
  if (pool == nullptr) {
    if (indexer_fast(s) && index_select_supported(false, s.n_entries)) {
      SelectArgs a = select_args(s, k_idx, s.n_entries, seqdiv(s), q_idx, w, n_valid, 1, k, idx_out, k, n_out, err);
      return cuda_status(launch_index_select(a, false, s.batch, s.n_entries, stream));
    }
    CSA2_TRY(do_index_flat(s, q_idx, w, k_idx, s.n_entries, seqdiv(s), n_valid, 1, ts, nullptr, nc, s.n_entries, err, stream));
    return do_topk(s, L, ws, ts, s.n_entries, nullptr, nc, s.n_entries, k, idx_out, nullptr, n_out, stream);
  }
  if (s.pool_blocks < 1 || n_pool == nullptr || s.n_entries % s.block != 0) return CSA2_ERR_INVALID_ARG;
  if (pooled_fast(s) && index_select_supported(true, s.pool_blocks)) {
    SelectArgs a = select_args(s, k_idx, s.n_entries, seqdiv(s), q_idx, w, n_valid, 1, k, idx_out, k, n_out, err);
    a.pool = pool;
    a.n_pool = n_pool;
    a.pool_cap = s.pool_blocks;
    return cuda_status(launch_index_select(a, true, s.batch, s.pool_blocks, stream));
  }
  CSA2_TRY(do_index_pooled(s, q_idx, w, k_idx, n_valid, pool, n_pool, ts, tc, nc, err, stream));
  const int64_t ld = int64_t(s.pool_blocks) * s.block;
  return do_topk(s, L, ws, ts, ld, tc, nc, ld, k, idx_out, nullptr, n_out, stream);
}

int csa2_topk(const csa2_shape* shape, const float* scores, int32_t ld, const int32_t* cand,
              const int32_t* n_cand, int32_t k, int32_t* idx_out, float* score_out, void* ws, size_t ws_bytes,
              csa2_stream_t stream) {
  CSA2_TRY(check_shape(shape));
  const csa2_shape& s = *shape;
  CSA2_TRY(check_ws(s, ws, ws_bytes));
  if (scores == nullptr || idx_out == nullptr || ld < 1 || k < 1) return CSA2_ERR_INVALID_ARG;
  if (k > topk_max_chunk() || ld > (1 << 28)) return CSA2_ERR_UNSUPPORTED;
  const WsLayout L = layout(s);
  // the chunk buffers are sized for the shape's longest candidate list and max(K, P)
  const int64_t maxc = topk_max_chunk();
  if (ld > maxc) {
    const int64_t chunks = ceil_div(ld, maxc);
    if (k > maxc / 2) return CSA2_ERR_UNSUPPORTED;   // merges must shrink the list
    if (chunks > L.tk_chunks || k > L.tk_kmax) return CSA2_ERR_WORKSPACE;
  }
  return do_topk(s, L, ws, scores, ld, cand, n_cand, ld, k, idx_out, score_out, nullptr, stream);
}

int csa2_sparse_attn(const csa2_shape* shape, const void* q, const void* k_main, const void* v_main,
                     const int32_t* idx, const void* k_swa, const void* v_swa, const int32_t* n_swa, float* out,
                     float* lse, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  CSA2_TRY(check_shape(shape));
  const csa2_shape& s = *shape;
  CSA2_TRY(check_ws(s, ws, ws_bytes));
  if (idx == nullptr) return CSA2_ERR_INVALID_ARG;
  CSA2_TRY(check_attn_args(s, q, k_main, v_main, out));
  CSA2_TRY(check_sswa(s, k_swa, v_swa, n_swa));
  const WsLayout L = layout(s);
  return do_attn(s, q, k_main, v_main, idx, k_swa, v_swa, n_swa, out, lse, at<int>(ws, L.hdr), stream);
}

int csa2_layer_group(const csa2_shape* shape, const csa2_layer* layers, int32_t n_layers, const void* k_main,
                     const void* v_main, const void* k_idx, const void* kb, const int32_t* n_valid,
                     const int32_t* n_swa, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  CSA2_TRY(check_shape(shape));
  const csa2_shape& s = *shape;
  CSA2_TRY(check_ws(s, ws, ws_bytes));
  if (layers == nullptr || n_layers < 1 || k_idx == nullptr || n_valid == nullptr) return CSA2_ERR_INVALID_ARG;
  if (indexer_fast(s) && !aligned16(k_idx)) return CSA2_ERR_INVALID_ARG;
  // validate the whole group before enqueueing anything
  bool have_idx = false;
  for (int l = 0; l < n_layers; ++l) {
    const csa2_layer& y = layers[l];
    if (y.mode != CSA2_FULL && y.mode != CSA2_REINDEX && y.mode != CSA2_REUSE && y.mode != CSA2_SWA)
      return CSA2_ERR_INVALID_ARG;
    if (y.hier != 0 && y.hier != 1) return CSA2_ERR_INVALID_ARG;
    CSA2_TRY(check_attn_args(s, y.q, k_main, v_main, y.out));
    CSA2_TRY(check_sswa(s, y.k_swa, y.v_swa, n_swa));
    if (y.mode == CSA2_SWA) {
      if (s.swa < 1) return CSA2_ERR_INVALID_ARG;
      continue;
    }
    if (y.mode == CSA2_REUSE) {
      if (!have_idx) return CSA2_ERR_INVALID_ARG;
      continue;
    }
    if (y.q_idx == nullptr || y.w_idx == nullptr) return CSA2_ERR_INVALID_ARG;
    if (y.hier) {
      if (kb == nullptr || s.pool_blocks < 1 || s.n_entries % s.block != 0) return CSA2_ERR_INVALID_ARG;
      if (indexer_fast(s) && !aligned16(kb)) return CSA2_ERR_INVALID_ARG;
    }
    have_idx = true;
  }
  const WsLayout L = layout(s);
  int* err = at<int>(ws, L.hdr);
  const int32_t* cur = nullptr;
  for (int l = 0; l < n_layers; ++l) {
    const csa2_layer& y = layers[l];
    // Another attention-only launch next (Reuse or SWA layer): release it at this
    // attention's end, unless the batch is small enough that both launches' CTAs
    // find SMs of their own (then its CTAs fetch their window rows early).
    const bool attn_next = l + 1 < n_layers && (layers[l + 1].mode == CSA2_REUSE || layers[l + 1].mode == CSA2_SWA) &&
                           !(attn_fast(s) && 2 * s.batch * attn_cluster(s.topk, s.swa) <= device_sm_count());
    if (y.mode == CSA2_SWA) {
      CSA2_TRY(do_attn(s, y.q, k_main, v_main, nullptr, y.k_swa, y.v_swa, n_swa, y.out, y.lse, err, stream, true,
                       attn_next));
      continue;
    }
    if (y.mode != CSA2_REUSE) {
      int32_t* dst = y.idx_out != nullptr ? y.idx_out : at<int32_t>(ws, L.idx);
      float* ts = at<float>(ws, L.tok_scores);
      int32_t* tc = at<int32_t>(ws, L.tok_cand);
      int32_t* nc = at<int32_t>(ws, L.n_cand);
      if (y.hier) {
        int32_t* pool = at<int32_t>(ws, L.pool);
        int32_t* npool = at<int32_t>(ws, L.n_pool);
        CSA2_TRY(do_index_blocks(s, L, ws, y.q_idx, y.w_idx, kb, n_valid, pool, npool, stream));
        if (pooled_fast(s) && index_select_supported(true, s.pool_blocks)) {
          // fused: pooled token scoring and Top-K in one cluster launch
          SelectArgs a = select_args(s, k_idx, s.n_entries, seqdiv(s), y.q_idx, y.w_idx, n_valid, 1, s.topk, dst, s.topk,
                                     nullptr, err);
          a.pool = pool;
          a.n_pool = npool;
          a.pool_cap = s.pool_blocks;
          CSA2_TRY(cuda_status(launch_index_select(a, true, s.batch, s.pool_blocks, stream)));
        } else {
          CSA2_TRY(do_index_pooled(s, y.q_idx, y.w_idx, k_idx, n_valid, pool, npool, ts, tc, nc, err, stream));
          const int64_t ld = int64_t(s.pool_blocks) * s.block;
          CSA2_TRY(do_topk(s, L, ws, ts, ld, tc, nc, ld, s.topk, dst, nullptr, nullptr, stream));
        }
      } else if (indexer_fast(s) && index_select_supported(false, s.n_entries)) {
        // fused: flat token scoring and Top-K in one cluster launch
        SelectArgs a = select_args(s, k_idx, s.n_entries, seqdiv(s), y.q_idx, y.w_idx, n_valid, 1, s.topk, dst, s.topk,
                                   nullptr, err);
        CSA2_TRY(cuda_status(launch_index_select(a, false, s.batch, s.n_entries, stream)));
      } else {
        CSA2_TRY(do_index_flat(s, y.q_idx, y.w_idx, k_idx, s.n_entries, seqdiv(s), n_valid, 1, ts, nullptr, nc, s.n_entries,
                               err, stream));
        CSA2_TRY(do_topk(s, L, ws, ts, s.n_entries, nullptr, nc, s.n_entries, s.topk, dst, nullptr, nullptr,
                         stream));
      }
      cur = dst;
    }
    CSA2_TRY(do_attn(s, y.q, k_main, v_main, cur, y.k_swa, y.v_swa, n_swa, y.out, y.lse, err, stream, false,
                     attn_next));
  }
  return CSA2_OK;
}

int csa2_shard_slice(const int32_t* ids, int32_t batch, int32_t ld, int32_t lo, int32_t hi, int32_t delta,
                     int32_t* out, int32_t ld_out, int32_t* n_out, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  if (ids == nullptr || out == nullptr || batch < 1 || ld < 1 || ld_out < 1 || lo > hi) return CSA2_ERR_INVALID_ARG;
  if (ld > (1 << 24) || ld_out > (1 << 24) || batch > (1 << 20)) return CSA2_ERR_UNSUPPORTED;
  if (int64_t(hi) + delta > INT32_MAX || int64_t(lo) + delta < INT32_MIN) return CSA2_ERR_INVALID_ARG;
  if (ws == nullptr || ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return CSA2_ERR_WORKSPACE;
  ShardSliceArgs a{};
  a.ids = ids;
  a.ld = ld;
  a.lo = lo;
  a.hi = hi;
  a.delta = delta;
  a.out = out;
  a.ld_out = ld_out;
  a.n_out = n_out;
  a.err = static_cast<int*>(ws);
  return cuda_status(launch_shard_slice(a, batch, stream));
}

int csa2_shard_counts(const int32_t* n_valid, int32_t batch, int32_t e0, int32_t n_loc, int32_t div, int32_t* out,
                      csa2_stream_t stream) {
  if (n_valid == nullptr || out == nullptr || batch < 1 || e0 < 0 || n_loc < 0 || div < 1) return CSA2_ERR_INVALID_ARG;
  return cuda_status(launch_shard_counts(n_valid, batch, e0, n_loc, div, out, stream));
}

int csa2_concat_parts(int32_t parts, int32_t batch, int32_t k, const int32_t* ids, const float* scores,
                      int32_t* ids_out, float* scores_out, csa2_stream_t stream) {
  if (parts < 1 || batch < 1 || k < 1 || ids == nullptr || ids_out == nullptr) return CSA2_ERR_INVALID_ARG;
  if (scores != nullptr && scores_out == nullptr) return CSA2_ERR_INVALID_ARG;
  if (int64_t(parts) * k > (1 << 28)) return CSA2_ERR_UNSUPPORTED;
  ConcatArgs a{};
  a.ids = ids;
  a.scores = scores;
  a.ids_out = ids_out;
  a.scores_out = scores_out;
  a.parts = parts;
  a.batch = batch;
  a.k = k;
  return cuda_status(launch_concat_parts(a, stream));
}

int csa2_merge_attn(int32_t parts, int32_t rows, int32_t v_dim, const float* out_parts, const float* lse_parts,
                    float* out, float* lse, csa2_stream_t stream) {
  if (parts < 1 || rows < 1 || v_dim < 1 || out_parts == nullptr || lse_parts == nullptr || out == nullptr)
    return CSA2_ERR_INVALID_ARG;
  if (parts > 1024 || v_dim > 1024 || int64_t(rows) * v_dim * parts > (int64_t(1) << 40)) return CSA2_ERR_UNSUPPORTED;
  MergeAttnArgs a{};
  a.out_parts = out_parts;
  a.lse_parts = lse_parts;
  a.out = out;
  a.lse = lse;
  a.parts = parts;
  a.rows = rows;
  a.v_dim = v_dim;
  return cuda_status(launch_merge_attn(a, stream));
}

const char* csa2_status_str(int status) {
  switch (status) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID_ARG: return "invalid argument (null/misaligned pointer, bad size or mode sequence)";
    case CSA2_ERR_UNSUPPORTED: return "unsupported shape";
    case CSA2_ERR_WORKSPACE: return "workspace too small or misaligned";
    case CSA2_ERR_CUDA: return "CUDA launch or runtime error";
    case CSA2_ERR_DEVICE_CHECK: return "a kernel recorded an out-of-range input";
    case CSA2_ERR_TIMEOUT: return "a bounded device wait gave up";
    default: return "unknown status";
  }
}

int csa2_read_device_error(void* ws, csa2_stream_t stream, int32_t* detail) {
  if (ws == nullptr) return CSA2_ERR_WORKSPACE;
  int host[2] = {0, 0};
  if (cudaMemcpyAsync(host, ws, sizeof(host), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return CSA2_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return CSA2_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(host), stream) != cudaSuccess) return CSA2_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return CSA2_ERR_CUDA;
  if (detail != nullptr) *detail = host[0] & 0xff;
  if (host[0] == 0) return CSA2_OK;
  return (host[0] & kErrTimeout) ? CSA2_ERR_TIMEOUT : CSA2_ERR_DEVICE_CHECK;
}

unsigned long long csa2_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int csa2_debug_wait_timeout(const csa2_shape* shape, const void* q_idx, const float* w, const void* k_idx,
                            const int32_t* n_valid, int32_t k, int32_t* idx_out, uint32_t wait_limit_ns, void* ws,
                            size_t ws_bytes, csa2_stream_t stream) {
  CSA2_TRY(check_shape(shape));
  const csa2_shape& s = *shape;
  CSA2_TRY(check_ws(s, ws, ws_bytes));
  if (q_idx == nullptr || w == nullptr || k_idx == nullptr || n_valid == nullptr || idx_out == nullptr || k < 1 ||
      k > s.topk)
    return CSA2_ERR_INVALID_ARG;
  if (wait_limit_ns < 1000u || wait_limit_ns > 100000000u) return CSA2_ERR_INVALID_ARG;
  if (!indexer_fast(s) || !index_select_supported(false, s.n_entries) || !aligned16(k_idx))
    return CSA2_ERR_UNSUPPORTED;
  const WsLayout L = layout(s);
  SelectArgs a = select_args(s, k_idx, s.n_entries, seqdiv(s), q_idx, w, n_valid, 1, k, idx_out, k, nullptr,
                             at<int>(ws, L.hdr));
  a.wait_ns = wait_limit_ns;
  a.skip_first_copy = 1;
  return cuda_status(launch_index_select(a, false, s.batch, s.n_entries, stream));
}

int csa2_fast_path(const csa2_shape* shape, int32_t* indexer_fast_out, int32_t* attention_fast_out) {
  if (check_shape(shape) != CSA2_OK) return 0;
  const int ix = indexer_fast(*shape) ? 1 : 0;
  const int at_ = attn_fast(*shape) ? 1 : 0;
  if (indexer_fast_out != nullptr) *indexer_fast_out = ix;
  if (attention_fast_out != nullptr) *attention_fast_out = at_;
  return ix && at_;
}

}  // extern "C"

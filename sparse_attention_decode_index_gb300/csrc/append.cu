// Decode-step cache maintenance: appending compressed entries to the main KV
// and indexer-key caches with incremental block summary keys, and pushing
// each decoded token into its query's SWA ring (DeepSeek V4.1 Flash
// architecture page: bullet "Hierarchical indexer" for the per-block summary
// keys, bullet "Sparse attention" for the 128-token SWA window).
//
// Both kernels run one CTA per query.  They move a few hundred bytes per
// query, so they are bound by launch latency, not bandwidth.  Neither lets the
// next launch in the stream start before it completes: the library's other
// kernels read inputs such as n_valid, n_swa and the SWA rows before waiting on
// the preceding launch, and these kernels write exactly those.
#include "common.cuh"
#include "internal.h"

namespace csa2 {

namespace {

constexpr int kThreads = 256;

// Copy `n` 16-bit units (the element types are bf16 or fp32, both whole
// multiples of 2 bytes).
__device__ __forceinline__ void copy_units(uint16_t* dst, const uint16_t* src, long long n) {
  for (long long i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
}

__global__ void __launch_bounds__(kThreads) kv_append_kernel(const KvAppendArgs a) {
  const int b = blockIdx.x;
  pdl_wait();   // no early trigger: the next launch may read what this one writes before its own wait
  const int units = a.dtype == 1 ? 2 : 1;   // 16-bit units per element
  const int nv0 = clamp_count(a.n_valid[b], a.n_entries, a.err);
  int m = clamp_count(a.n_new[b], a.max_new, a.err);
  if (nv0 + m > a.n_entries) {
    if (threadIdx.x == 0) report(a.err, kErrBadCount, nv0 + m);
    m = a.n_entries - nv0;
  }
  // rows j < m of the new entries are contiguous, and so are their destinations
  const long long src_row = (long long)b * a.max_new, dst_row = (long long)b * a.n_entries + nv0;
  copy_units(static_cast<uint16_t*>(a.k_main) + dst_row * a.k_dim * units,
             static_cast<const uint16_t*>(a.k_new) + src_row * a.k_dim * units, (long long)m * a.k_dim * units);
  copy_units(static_cast<uint16_t*>(a.v_main) + dst_row * a.v_dim * units,
             static_cast<const uint16_t*>(a.v_new) + src_row * a.v_dim * units, (long long)m * a.v_dim * units);
  copy_units(static_cast<uint16_t*>(a.k_idx) + dst_row * a.idx_dim * units,
             static_cast<const uint16_t*>(a.kidx_new) + src_row * a.idx_dim * units,
             (long long)m * a.idx_dim * units);
  __syncthreads();   // the new indexer keys are visible to every thread of the CTA
  const int nv1 = nv0 + m;
  if (a.kb != nullptr && m > 0) {
    const int j0 = nv0 / a.block, j1 = (nv1 - 1) / a.block;   // blocks the new positions touch
    const int n = (j1 - j0 + 1) * a.idx_dim;
    for (int e = threadIdx.x; e < n; e += blockDim.x) {
      const int j = j0 + e / a.idx_dim, d = e % a.idx_dim;
      const float v = block_key_elem(a.k_idx, (long long)b * a.n_entries, a.idx_dim, a.block, nv1, j, d, a.dtype,
                                     a.round_to_int);
      store_elem(a.kb, ((long long)b * a.nb_cap + j) * a.idx_dim + d, a.dtype, v);
    }
  }
  __syncthreads();   // every thread read n_valid[b] before it changes
  if (threadIdx.x == 0) a.n_valid[b] = nv1;
}

__global__ void __launch_bounds__(kThreads) swa_append_kernel(const SwaAppendArgs a) {
  const int b = blockIdx.x;
  pdl_wait();   // no early trigger: the next launch may read what this one writes before its own wait
  const int units = a.dtype == 1 ? 2 : 1;
  int slot = a.head[b];
  if (slot < 0 || slot >= a.swa) {
    if (threadIdx.x == 0) report(a.err, kErrBadCount, slot);
    slot = slot < 0 ? 0 : a.swa - 1;
  }
  const int n = clamp_count(a.n_swa[b], a.swa, a.err);
  const long long row = (long long)b * a.swa + slot;
  for (int l = 0; l < a.n_layers; ++l) {
    const SwaAppendArgs::Slot& y = a.slot[l];
    copy_units(static_cast<uint16_t*>(y.k_swa) + row * a.k_dim * units,
               static_cast<const uint16_t*>(y.k_tok) + (long long)b * a.k_dim * units, (long long)a.k_dim * units);
    copy_units(static_cast<uint16_t*>(y.v_swa) + row * a.v_dim * units,
               static_cast<const uint16_t*>(y.v_tok) + (long long)b * a.v_dim * units, (long long)a.v_dim * units);
  }
  __syncthreads();   // every thread read head[b] and n_swa[b] before they change
  if (threadIdx.x == 0) {
    a.head[b] = slot + 1 == a.swa ? 0 : slot + 1;
    a.n_swa[b] = n < a.swa ? n + 1 : a.swa;
  }
}

}  // namespace

cudaError_t launch_kv_append(const KvAppendArgs& a, int batch, cudaStream_t st) {
  if (batch == 0) return cudaSuccess;
  note_launch();
  return launch_pdl(kv_append_kernel, dim3(unsigned(batch)), dim3(kThreads), 0, st, 1, a);
}

cudaError_t launch_swa_append(const SwaAppendArgs& a, int batch, cudaStream_t st) {
  if (batch == 0) return cudaSuccess;
  note_launch();
  return launch_pdl(swa_append_kernel, dim3(unsigned(batch)), dim3(kThreads), 0, st, 1, a);
}

}  // namespace csa2

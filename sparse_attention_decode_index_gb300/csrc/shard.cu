// Context-parallel helpers: one long sequence's compressed entries split by
// block-aligned ranges over several ranks (each rank holds entries
// [e0, e0 + n_loc) of every sequence of the batch).  Selection stays exact
// because the Top-k order (score descending, id ascending) is a strict total
// order: the global Top-k of a union is the Top-k of the union of each part's
// Top-k.  Attention stays exact up to rounding because softmax partials over
// disjoint key sets combine by their log-sum-exp.  (Architecture page
// k-a.in "DeepSeek V4.1 Flash", bullet "Hierarchical indexer": at most 16,384
// candidates whatever the context length; bullet "Sparse attention".)
//
//   shard_slice_kernel  -- the ids of a row that fall in [lo, hi), in their
//                          order, shifted by delta and compacted; -1 padded
//   shard_counts_kernel -- a rank's valid entries (or blocks): ceil(clamp(n_valid - e0, 0, n_loc) / div)
//   concat_parts_kernel -- the parts' (id, score) lists of each row side by side
//   merge_attn_kernel   -- softmax partials of G ranks combined in rank order
#include "common.cuh"
#include "internal.h"

// The helper kernels wait for the preceding launch and let their dependents in
// only when they complete (no early trigger): a following kernel may read the
// lists and counts they write before its own wait.

namespace csa2 {

namespace {

constexpr int kSliceThreads = 256;

__global__ void __launch_bounds__(kSliceThreads) shard_slice_kernel(const ShardSliceArgs a) {
  __shared__ int warp_tot[kSliceThreads / 32];
  __shared__ int base;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  const int* in = a.ids + (long long)b * a.ld;
  int* out = a.out + (long long)b * a.ld_out;
  if (tid == 0) base = 0;
  __syncthreads();
  for (int p0 = 0; p0 < a.ld; p0 += kSliceThreads) {
    const int p = p0 + tid;
    const int id = p < a.ld ? in[p] : -1;
    const bool keep = id >= 0 && id >= a.lo && id < a.hi;   // -1 pads are never kept
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) warp_tot[warp] = __popc(m);
    __syncthreads();
    int before = base;
    for (int w = 0; w < warp; ++w) before += warp_tot[w];
    const int slot = before + __popc(m & ((1u << lane) - 1u));
    if (keep && slot < a.ld_out) out[slot] = id + a.delta;
    __syncthreads();
    if (tid == 0) {
      int t = 0;
      for (int w = 0; w < kSliceThreads / 32; ++w) t += warp_tot[w];
      base += t;
    }
    __syncthreads();
  }
  const int n = base;
  if (n > a.ld_out && tid == 0) report(a.err, kErrBadCount, n);
  for (int p = n + tid; p < a.ld_out; p += kSliceThreads) out[p] = -1;
  if (tid == 0 && a.n_out != nullptr) a.n_out[b] = int(min((long long)n, a.ld_out));
}

__global__ void __launch_bounds__(256) shard_counts_kernel(const int* n_valid, int batch, int e0, int n_loc,
                                                           int div, int* out) {
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch) out[b] = (min(max(n_valid[b] - e0, 0), n_loc) + div - 1) / div;
}

// Rows of the parts' lists side by side: out[b, g * k + p] = in[g, b, p].
__global__ void __launch_bounds__(256) concat_parts_kernel(const ConcatArgs a) {
  pdl_wait();
  const long long n = (long long)a.parts * a.batch * a.k;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int p = int(i % a.k);
    const long long r = i / a.k;
    const int b = int(r % a.batch), g = int(r / a.batch);
    const long long o = ((long long)b * a.parts + g) * a.k + p;
    a.ids_out[o] = a.ids[i];
    if (a.scores != nullptr) a.scores_out[o] = a.scores[i];
  }
}

// One warp per (query, head): weights exp(lse_g - M) over the parts in rank
// order, then each lane combines dv / 32 columns.
__global__ void __launch_bounds__(256) merge_attn_kernel(const MergeAttnArgs a) {
  pdl_wait();
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);   // b * heads + h
  const int lane = threadIdx.x & 31;
  if (row >= a.rows) return;
  float M = -INFINITY;
  for (int g = 0; g < a.parts; ++g) M = fmaxf(M, a.lse_parts[(long long)g * a.rows + row]);
  float S = 0.f;
  for (int g = 0; g < a.parts; ++g) {
    const float l = a.lse_parts[(long long)g * a.rows + row];
    if (l != -INFINITY) S += expf(l - M);
  }
  const float inv = S > 0.f ? 1.f / S : 0.f;
  for (int d = lane; d < a.v_dim; d += 32) {
    float acc = 0.f;
    for (int g = 0; g < a.parts; ++g) {
      const float l = a.lse_parts[(long long)g * a.rows + row];
      if (l == -INFINITY) continue;
      acc += expf(l - M) * a.out_parts[((long long)g * a.rows + row) * a.v_dim + d];
    }
    a.out[(long long)row * a.v_dim + d] = acc * inv;
  }
  if (lane == 0 && a.lse != nullptr) a.lse[row] = M == -INFINITY ? -INFINITY : M + logf(S);
}

}  // namespace

cudaError_t launch_shard_slice(const ShardSliceArgs& a, int batch, cudaStream_t st) {
  if (batch == 0) return cudaSuccess;
  note_launch();
  return launch_pdl(shard_slice_kernel, dim3(unsigned(batch)), dim3(kSliceThreads), 0, st, 1, a);
}

cudaError_t launch_shard_counts(const int* n_valid, int batch, int e0, int n_loc, int div, int* out,
                                cudaStream_t st) {
  if (batch == 0) return cudaSuccess;
  note_launch();
  return launch_pdl(shard_counts_kernel, dim3(unsigned((batch + 255) / 256)), dim3(256), 0, st, 1, n_valid, batch,
                    e0, n_loc, div, out);
}

cudaError_t launch_concat_parts(const ConcatArgs& a, cudaStream_t st) {
  const long long n = (long long)a.parts * a.batch * a.k;
  if (n == 0) return cudaSuccess;
  note_launch();
  const unsigned grid = unsigned(min((n + 255) / 256, (long long)4096));
  return launch_pdl(concat_parts_kernel, dim3(grid), dim3(256), 0, st, 1, a);
}

cudaError_t launch_merge_attn(const MergeAttnArgs& a, cudaStream_t st) {
  if (a.rows == 0) return cudaSuccess;
  note_launch();
  return launch_pdl(merge_attn_kernel, dim3(unsigned((a.rows + 7) / 8)), dim3(256), 0, st, 1, a);
}

}  // namespace csa2

// Exact Top-K selection under the total order (score descending, index
// ascending), output in ascending index order and padded with -1.
// (DeepSeek V4.1 Flash architecture page, bullet "Sparse attention": each
// query reads its Top-512 main-KV entries; bullet "Hierarchical indexer":
// the block pool.  The pages do not state a tie rule; the lowest index wins.)
//
// One CTA selects the Top-k of one chunk of up to 16,384 positions:
//   1. scores are mapped to order-preserving uint32 keys held in registers;
//   2. radix select narrows a key interval [lo, hi] that contains the k-th
//      largest key: each pass histograms the keys of the interval into 2048
//      power-of-two-wide bins and keeps the bin where the count from the top
//      reaches k (at most three passes for 32-bit keys);
//   3. with the threshold key T known, a single block-wide scan over
//      (count > T, count == T) in position order places every key > T and
//      the first (k - #>T) keys == T at their output slots.
// Larger inputs are split into chunks whose Top-k lists are merged by a
// further pass over the concatenated lists (exact: a global Top-k member is
// in its chunk's Top-k under a strict total order).
#include "common.cuh"
#include "internal.h"

namespace csa2 {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kBinsPerThread = kBins / kThreads;   // 4

struct TopkSmem {
  uint32_t hist[kBins];
  uint32_t warp_a[kWarps];
  uint32_t warp_b[kWarps];
  uint32_t sel_bin;
  uint32_t sel_above;
};

// Exclusive block-wide sum; also returns the total.  Ends with a barrier so the
// scratch can be reused immediately.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* scratch, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = lane < kWarps ? scratch[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kWarps) scratch[lane] = s;
  }
  __syncthreads();
  const uint32_t before = warp > 0 ? scratch[warp - 1] : 0u;
  total = scratch[kWarps - 1];
  __syncthreads();
  return before + x - v;
}

__device__ __forceinline__ uint32_t block_sum(uint32_t v, uint32_t* scratch) {
  uint32_t total;
  block_excl_scan(v, scratch, total);
  return total;
}

__device__ __forceinline__ void block_minmax(uint32_t& lo, uint32_t& hi, uint32_t* sa, uint32_t* sb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if (lane == 0) {
    sa[warp] = lo;
    sb[warp] = hi;
  }
  __syncthreads();
  lo = sa[0];
  hi = sb[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) {
    lo = min(lo, sa[w]);
    hi = max(hi, sb[w]);
  }
  __syncthreads();
}

template <int IPT>
__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkArgs a) {
  __shared__ TopkSmem sm;
  const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  const int chunks = gridDim.x;
  const long long row = (long long)b * a.ld_in;
  int n = a.n_cand != nullptr ? clamp_count(a.n_cand[b], a.n_cap, a.err) : a.n_fixed;
  const int base = c * a.chunk;                       // first position of this chunk
  const int len = max(0, min(a.chunk, n - base));     // positions in this chunk
  const int p0 = tid * IPT;                           // first local position of this thread

  // Independent, vectorised loads of this thread's IPT scores (and candidate ids).
  uint32_t key[IPT];
  uint32_t valid = 0;
  const float* sp = a.scores + row + base + p0;
  const int* cp = a.cand != nullptr ? a.cand + row + base + p0 : nullptr;
  const int nloc = max(0, min(IPT, len - p0));
  float sv[IPT];
  int cv[IPT];
  const bool vec = nloc == IPT &&
                   ((reinterpret_cast<uintptr_t>(sp) | reinterpret_cast<uintptr_t>(cp)) & 15u) == 0;
  if (vec) {
#pragma unroll
    for (int i = 0; i < IPT; i += 4) {
      const float4 v = *reinterpret_cast<const float4*>(sp + i);
      sv[i] = v.x; sv[i + 1] = v.y; sv[i + 2] = v.z; sv[i + 3] = v.w;
    }
    if (cp != nullptr) {
#pragma unroll
      for (int i = 0; i < IPT; i += 4) {
        const int4 v = *reinterpret_cast<const int4*>(cp + i);
        cv[i] = v.x; cv[i + 1] = v.y; cv[i + 2] = v.z; cv[i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < IPT; ++i) cv[i] = 0;
    }
  } else {
#pragma unroll
    for (int i = 0; i < IPT; ++i) {
      sv[i] = i < nloc ? sp[i] : 0.f;
      cv[i] = (cp != nullptr && i < nloc) ? cp[i] : 0;
    }
  }
#pragma unroll
  for (int i = 0; i < IPT; ++i) {
    const bool ok = i < nloc && cv[i] >= 0;
    key[i] = ok ? score_key(sv[i]) : 0u;
    valid |= ok ? (1u << i) : 0u;
  }
  const uint32_t n_valid = block_sum(__popc(valid), sm.warp_a);
  const uint32_t k = uint32_t(a.k);

  uint32_t T = 0u, need_eq = 0u;
  bool take_all = n_valid <= k;
  if (!take_all) {
    uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
    for (int i = 0; i < IPT; ++i)
      if (valid & (1u << i)) {
        lo = min(lo, key[i]);
        hi = max(hi, key[i]);
      }
    block_minmax(lo, hi, sm.warp_a, sm.warp_b);
    uint32_t above = 0u;                               // keys > hi (already selected)
    while (lo != hi) {
      const uint32_t range = hi - lo;
      const int bits = 32 - __clz(range);
      const int shift = bits > 11 ? bits - 11 : 0;
      for (int j = tid; j < kBins; j += kThreads) sm.hist[j] = 0u;
      __syncthreads();
#pragma unroll
      for (int i = 0; i < IPT; ++i)
        if ((valid & (1u << i)) && key[i] >= lo && key[i] <= hi) atomicAdd(&sm.hist[(key[i] - lo) >> shift], 1u);
      __syncthreads();
      // thread t owns bins kBins-1-4t .. kBins-4-4t, scanned from the top
      uint32_t cnt[kBinsPerThread];
      uint32_t local = 0u;
#pragma unroll
      for (int j = 0; j < kBinsPerThread; ++j) {
        cnt[j] = sm.hist[kBins - 1 - tid * kBinsPerThread - j];
        local += cnt[j];
      }
      uint32_t tot;
      uint32_t before = above + block_excl_scan(local, sm.warp_a, tot);
#pragma unroll
      for (int j = 0; j < kBinsPerThread; ++j) {
        if (before < k && before + cnt[j] >= k) {
          sm.sel_bin = uint32_t(kBins - 1 - tid * kBinsPerThread - j);
          sm.sel_above = before;
        }
        before += cnt[j];
      }
      __syncthreads();
      const uint32_t bin = sm.sel_bin;
      above = sm.sel_above;
      const uint32_t nlo = lo + (bin << shift);
      const uint32_t width = (1u << shift) - 1u;
      hi = (hi - nlo > width) ? nlo + width : hi;
      lo = nlo;
      __syncthreads();
    }
    T = lo;
    need_eq = k - above;
  }

  // Final placement in position order.
  uint32_t n_gt = 0u, n_eq = 0u;
#pragma unroll
  for (int i = 0; i < IPT; ++i) {
    if (!(valid & (1u << i))) continue;
    if (take_all || key[i] > T)
      ++n_gt;
    else if (key[i] == T)
      ++n_eq;
  }
  uint32_t tot;
  const uint32_t packed = block_excl_scan((n_gt << 16) | n_eq, sm.warp_a, tot);
  uint32_t gt_before = packed >> 16, eq_before = packed & 0xffffu;
  uint32_t slot = gt_before + min(eq_before, need_eq);
  const long long out = ((long long)b * chunks + c) * a.k;
#pragma unroll
  for (int i = 0; i < IPT; ++i) {
    if (!(valid & (1u << i))) continue;
    bool take = false;
    if (take_all || key[i] > T) {
      take = true;
    } else if (key[i] == T) {
      take = eq_before < need_eq;
      ++eq_before;
    }
    if (take) {
      const long long pos = base + p0 + i;
      a.idx_out[out + slot] = a.cand != nullptr ? a.cand[row + pos] : int(pos);
      if (a.score_out != nullptr) a.score_out[out + slot] = key_score(key[i]);
      ++slot;
    }
  }
  const int selected = int(min(n_valid, k));
  if (a.n_out != nullptr && chunks == 1 && tid == 0) a.n_out[b] = selected;
  for (int j = selected + tid; j < a.k; j += kThreads) {
    a.idx_out[out + j] = -1;
    if (a.score_out != nullptr) a.score_out[out + j] = -__int_as_float(0x7f800000);
  }
}

}  // namespace

int topk_max_chunk() { return kThreads * 32; }

cudaError_t launch_topk(const TopkArgs& a, int chunks, int batch, cudaStream_t st) {
  if (batch == 0 || chunks == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(chunks), static_cast<unsigned>(batch));
  note_launch();
  if (a.chunk <= kThreads * 8)
    topk_kernel<8><<<grid, kThreads, 0, st>>>(a);
  else
    topk_kernel<32><<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace csa2

// Exact Top-K selection under the total order (score descending, index
// ascending), output in ascending index order and padded with -1.
// (DeepSeek V4.1 Flash architecture page, bullet "Sparse attention": each
// query reads its Top-512 main-KV entries; bullet "Hierarchical indexer":
// the block pool.  The pages do not state a tie rule; the lowest index wins.)
//
// One CTA selects the Top-k of one chunk of up to 16,384 positions:
//   1. scores are mapped to order-preserving uint32 keys held in registers;
//   2. radix select narrows a key interval [lo, hi] that contains the k-th
//      largest key: each pass histograms the keys of the interval into 256
//      power-of-two-wide bins and keeps the bin where the count from the top
//      reaches k (at most four passes for 32-bit keys).  The histogram keeps one
//      counter per (bin, lane), so the lanes of a warp never contend for a
//      counter or a bank even when integer-valued scores crowd into one bin;
//   3. with T known, a single block-wide scan over (count > T, count == T) in
//      position order places every key > T and the first (k - #>T) keys == T
//      at their output slots.
// Larger inputs are split into chunks whose Top-k lists are merged by a
// further pass over the concatenated lists (exact: a global Top-k member is
// in its chunk's Top-k under a strict total order).
#include "common.cuh"
#include "internal.h"

namespace csa2 {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

constexpr int kBins = 256;                         // 8-bit digits

struct TopkSmem {
  uint32_t hist[kBins][32];                        // [bin][lane] private counters
  uint32_t tot[kBins];
  uint32_t warp_a[kWarps];
  uint32_t warp_b[kWarps];
  uint32_t sel_bin;
  uint32_t sel_above;
};

// Exclusive block-wide sum; also returns the total.  Ends with a barrier so the
// scratch can be reused immediately.
template <int NW = kWarps>
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
    uint32_t s = lane < NW ? scratch[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < NW) scratch[lane] = s;
  }
  __syncthreads();
  const uint32_t before = warp > 0 ? scratch[warp - 1] : 0u;
  total = scratch[NW - 1];
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

// Two CTAs per SM (64 registers, a few hundred bytes of spills at IPT = 32):
// the 1M decoder group's 256 chunk CTAs then run in one wave instead of 1.7
// (measured 565.3 -> 562.9 us per group step).
template <int IPT>
__global__ void __launch_bounds__(kThreads, 2) topk_kernel(const TopkArgs a) {
  __shared__ TopkSmem sm;
  const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  pdl_launch_dependents();
  pdl_wait();   // scores / candidates come from the preceding launch
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
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t above = 0u;                               // keys > hi (already selected)
    while (lo != hi) {
      const uint32_t range = hi - lo;
      const int bits = 32 - __clz(range);
      const int shift = bits > 8 ? bits - 8 : 0;
      uint4* hv = reinterpret_cast<uint4*>(&sm.hist[0][0]);
      for (int j = tid; j < kBins * 32 / 4; j += kThreads) hv[j] = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
#pragma unroll
      for (int i = 0; i < IPT; ++i)
        if ((valid & (1u << i)) && key[i] >= lo && key[i] <= hi) atomicAdd(&sm.hist[(key[i] - lo) >> shift][lane], 1u);
      __syncthreads();
      // bin totals: thread t < 256 sums the 32 lane counters of bin t (rotated: no bank conflicts)
      if (tid < kBins) {
        uint32_t v = 0u;
#pragma unroll
        for (int l = 0; l < 32; ++l) v += sm.hist[tid][(l + tid) & 31];
        sm.tot[tid] = v;
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns bins 255 - 8l .. 248 - 8l, scanned from the top
        uint32_t cnt[8], local = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          cnt[j] = sm.tot[kBins - 1 - lane * 8 - j];
          local += cnt[j];
        }
        uint32_t incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        uint32_t before = above + incl - local;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (before < k && before + cnt[j] >= k) {
            sm.sel_bin = uint32_t(kBins - 1 - lane * 8 - j);
            sm.sel_above = before;
          }
          before += cnt[j];
        }
      }
      __syncthreads();
      const uint32_t bin = sm.sel_bin;
      above = sm.sel_above;
      const uint32_t nlo = lo + (bin << shift);
      const uint32_t width = (1u << shift) - 1u;
      hi = (hi - nlo > width) ? nlo + width : hi;
      lo = nlo;
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


// ---------------------------------------------------------------------------
// Cluster Top-k: one thread-block cluster of C CTAs (C <= 8) per row.  CTA c
// holds positions [c * chunk, (c + 1) * chunk) in registers; every radix pass
// builds a local 256-bin histogram (lane-private counters), publishes its bin
// totals in shared memory, and after one cluster barrier every CTA sums the C
// totals through distributed shared memory and picks the same bin.  The tie
// quota and the output offset of each CTA follow from a prefix over the CTAs'
// (count > T, count == T), so the output is the same as the single-CTA kernel.

constexpr int kCThreads = 256;
constexpr int kCWarps = kCThreads / 32;
constexpr int kMaxCluster = 8;

struct ClusterTopkSmem {
  uint32_t hist[kBins][32];
  uint32_t tot[2][kBins];      // this CTA's bin totals (double-buffered across passes)
  uint32_t gtot[kBins];        // cluster-wide totals
  uint32_t stats[3];           // this CTA: valid count, min key, max key
  uint32_t fin[2];             // this CTA: count > T, count == T
  uint32_t red[2][kCWarps];
  uint32_t sel_bin, sel_above, lo, hi, n_valid, offset, quota;
};

template <int IPT>
__global__ void __launch_bounds__(kCThreads) topk_cluster_kernel(const TopkArgs a) {
  __shared__ ClusterTopkSmem sm;
  const int b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t crank = cluster_rank(), ncta = cluster_size();
  pdl_launch_dependents();
  pdl_wait();   // scores / candidates come from the preceding launch
  const long long row = (long long)b * a.ld_in;
  const int n = a.n_cand != nullptr ? clamp_count(a.n_cand[b], a.n_cap, a.err) : a.n_fixed;
  const int base = int(crank) * a.chunk;
  const int len = max(0, min(a.chunk, n - base));
  const int p0 = tid * IPT;

  uint32_t key[IPT];
  uint32_t valid = 0;
  {
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
  }

  // ---- local (count, min, max) -> cluster-wide
  {
    uint32_t cnt = __popc(valid), lo = 0xffffffffu, hi = 0u;
#pragma unroll
    for (int i = 0; i < IPT; ++i)
      if (valid & (1u << i)) {
        lo = min(lo, key[i]);
        hi = max(hi, key[i]);
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
      sm.red[0][warp] = lo;
      sm.red[1][warp] = hi;
      sm.hist[0][warp] = cnt;     // scratch before the histogram is used
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t c = 0, l = 0xffffffffu, h = 0u;
      for (int w = 0; w < kCWarps; ++w) {
        c += sm.hist[0][w];
        l = min(l, sm.red[0][w]);
        h = max(h, sm.red[1][w]);
      }
      sm.stats[0] = c;
      sm.stats[1] = l;
      sm.stats[2] = h;
    }
    cluster_sync_all();
    if (tid == 0) {
      uint32_t c = 0, l = 0xffffffffu, h = 0u;
      for (uint32_t r = 0; r < ncta; ++r) {
        const uint32_t rc = __float_as_uint(dsmem_ld_f32(dsmem_addr(&sm.stats[0], r)));
        const uint32_t rl = __float_as_uint(dsmem_ld_f32(dsmem_addr(&sm.stats[1], r)));
        const uint32_t rh = __float_as_uint(dsmem_ld_f32(dsmem_addr(&sm.stats[2], r)));
        c += rc;
        if (rc > 0) {
          l = min(l, rl);
          h = max(h, rh);
        }
      }
      sm.n_valid = c;
      sm.lo = l;
      sm.hi = h;
    }
    __syncthreads();
  }
  const uint32_t n_valid = sm.n_valid;
  const uint32_t k = uint32_t(a.k);
  const bool take_all = n_valid <= k;
  uint32_t T = 0u, need_eq = 0u;
  if (!take_all) {
    uint32_t lo = sm.lo, hi = sm.hi, above = 0u;
    int buf = 0;
    while (lo != hi) {
      const uint32_t range = hi - lo;
      const int bits = 32 - __clz(range);
      const int shift = bits > 8 ? bits - 8 : 0;
      uint4* hv = reinterpret_cast<uint4*>(&sm.hist[0][0]);
      for (int j = tid; j < kBins * 32 / 4; j += kCThreads) hv[j] = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
#pragma unroll
      for (int i = 0; i < IPT; ++i)
        if ((valid & (1u << i)) && key[i] >= lo && key[i] <= hi) atomicAdd(&sm.hist[(key[i] - lo) >> shift][lane], 1u);
      __syncthreads();
      {
        uint32_t v = 0u;
#pragma unroll
        for (int l = 0; l < 32; ++l) v += sm.hist[tid][(l + tid) & 31];
        sm.tot[buf][tid] = v;
      }
      cluster_sync_all();
      {
        uint32_t v = 0u;
        for (uint32_t r = 0; r < ncta; ++r) v += __float_as_uint(dsmem_ld_f32(dsmem_addr(&sm.tot[buf][tid], r)));
        sm.gtot[tid] = v;
      }
      __syncthreads();
      if (warp == 0) {
        uint32_t cnt[8], local = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          cnt[j] = sm.gtot[kBins - 1 - lane * 8 - j];
          local += cnt[j];
        }
        uint32_t incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        uint32_t before = above + incl - local;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (before < k && before + cnt[j] >= k) {
            sm.sel_bin = uint32_t(kBins - 1 - lane * 8 - j);
            sm.sel_above = before;
          }
          before += cnt[j];
        }
      }
      __syncthreads();
      const uint32_t bin = sm.sel_bin;
      above = sm.sel_above;
      const uint32_t nlo = lo + (bin << shift);
      const uint32_t width = (1u << shift) - 1u;
      hi = (hi - nlo > width) ? nlo + width : hi;
      lo = nlo;
      buf ^= 1;
    }
    T = lo;
    need_eq = k - above;
  }

  // ---- this CTA's (count > T, count == T), then its tie quota and output offset
  uint32_t n_gt = 0u, n_eq = 0u;
#pragma unroll
  for (int i = 0; i < IPT; ++i) {
    if (!(valid & (1u << i))) continue;
    if (take_all || key[i] > T)
      ++n_gt;
    else if (key[i] == T)
      ++n_eq;
  }
  {
    uint32_t g = n_gt, e = n_eq;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      g += __shfl_xor_sync(0xffffffffu, g, o);
      e += __shfl_xor_sync(0xffffffffu, e, o);
    }
    if (lane == 0) {
      sm.red[0][warp] = g;
      sm.red[1][warp] = e;
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t gg = 0, ee = 0;
      for (int w = 0; w < kCWarps; ++w) {
        gg += sm.red[0][w];
        ee += sm.red[1][w];
      }
      sm.fin[0] = gg;
      sm.fin[1] = ee;
    }
    cluster_sync_all();
    if (tid == 0) {
      uint32_t off = 0, eq_before = 0;
      for (uint32_t r = 0; r < crank; ++r) {
        const uint32_t rg = __float_as_uint(dsmem_ld_f32(dsmem_addr(&sm.fin[0], r)));
        const uint32_t re = __float_as_uint(dsmem_ld_f32(dsmem_addr(&sm.fin[1], r)));
        const uint32_t q = min(re, need_eq > eq_before ? need_eq - eq_before : 0u);
        off += rg + q;
        eq_before += re;
      }
      sm.offset = off;
      sm.quota = min(sm.fin[1], need_eq > eq_before ? need_eq - eq_before : 0u);
    }
    __syncthreads();
  }
  const uint32_t quota = sm.quota;
  uint32_t tot;
  const uint32_t packed = block_excl_scan<kCWarps>((n_gt << 16) | n_eq, sm.red[0], tot);
  uint32_t eq_before = packed & 0xffffu;
  uint32_t slot = sm.offset + (packed >> 16) + min(eq_before, quota);
  const long long out = (long long)b * a.k;
#pragma unroll
  for (int i = 0; i < IPT; ++i) {
    if (!(valid & (1u << i))) continue;
    bool take = false;
    if (take_all || key[i] > T) {
      take = true;
    } else if (key[i] == T) {
      take = eq_before < quota;
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
  if (crank == 0) {
    if (a.n_out != nullptr && tid == 0) a.n_out[b] = selected;
    for (int j = selected + tid; j < a.k; j += kCThreads) {
      a.idx_out[out + j] = -1;
      if (a.score_out != nullptr) a.score_out[out + j] = -__int_as_float(0x7f800000);
    }
  }
  cluster_sync_all();   // no CTA leaves while another may still read its shared memory
}

}  // namespace

int topk_max_chunk() { return kThreads * 32; }
int topk_cluster_max() { return kMaxCluster * kCThreads * 16; }

cudaError_t launch_topk_cluster(const TopkArgs& in, int batch, cudaStream_t st) {
  if (batch == 0) return cudaSuccess;
  TopkArgs a = in;
  const int n = a.n_cap;
  const int per_cta_max = kCThreads * 16;
  int c = (n + per_cta_max - 1) / per_cta_max;
  const int fill = (2 * device_sm_count()) / batch;   // aim for ~2 CTAs per SM
  if (c < fill) c = fill;
  if (c > kMaxCluster) c = kMaxCluster;
  if (c < 1) c = 1;
  int chunk = (n + c - 1) / c;
  chunk = (chunk + 3) / 4 * 4;
  if (chunk < 4) chunk = 4;
  c = (n + chunk - 1) / chunk;
  if (c < 1) c = 1;
  a.chunk = chunk;
  note_launch();
  const dim3 grid(static_cast<unsigned>(c), static_cast<unsigned>(batch));
  if (chunk <= kCThreads * 4) return launch_pdl(topk_cluster_kernel<4>, grid, dim3(kCThreads), 0, st, unsigned(c), a);
  if (chunk <= kCThreads * 8) return launch_pdl(topk_cluster_kernel<8>, grid, dim3(kCThreads), 0, st, unsigned(c), a);
  return launch_pdl(topk_cluster_kernel<16>, grid, dim3(kCThreads), 0, st, unsigned(c), a);
}

cudaError_t launch_topk(const TopkArgs& a, int chunks, int batch, cudaStream_t st) {
  if (batch == 0 || chunks == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(chunks), static_cast<unsigned>(batch));
  note_launch();
  if (a.chunk <= kThreads * 8) return launch_pdl(topk_kernel<8>, grid, dim3(kThreads), 0, st, 1, a);
  return launch_pdl(topk_kernel<32>, grid, dim3(kThreads), 0, st, 1, a);
}

}  // namespace csa2
